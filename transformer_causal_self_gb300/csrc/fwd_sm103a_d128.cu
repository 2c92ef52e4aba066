// Causal GQA attention prefill for head size 128, bf16 in / bf16 out, fp32
// accumulation, for sm_103a (tcgen05 MMAs with TMEM accumulators, TMA tiles,
// online softmax in fp32).  The T x T score matrix never leaves the SM
// ("Grasping Codes and Math 02", section "Flash Attention: The GPU Does
// Everything in One Pass").  The unit schedule (two query tiles A and B per
// unit that read the same KV head) is in fwd_units.cuh.
//
// The second GEMM is computed transposed and shared by both query tiles:
//
//   O^T[c, q] += sum_k V[k, c] P[q, k]   over the 256 queries of tiles A and B
//
// one M=128 (channels) x N=256 (queries) x K=16 (keys) MMA per 16 keys.  On
// this part an N=128 MMA takes about as much tensor time as an N=256 one, so
// this halves the cost of P V against O = P V per tile (N = 128).  P goes
// through shared memory (rows 0-127 tile A, 128-255 tile B, K-major, 128-byte
// swizzle); V is read MN-major as the A operand.  S = Q K^T stays N=128 per
// tile: TMEM holds S_A [0,128), S_B [128,256) and O^T [256,512) with lanes =
// channels and columns = queries (tile A 0-127, tile B 128-255).
//
// Warp roles (384 threads; setmaxnreg: 200 registers for the softmax
// warpgroups, 104 for the third):
//   warps 0-3   softmax of tile A: thread = query row = TMEM lane of S_A, and
//               channel of O^T for the lazy rescale and the epilogue
//   warps 4-7   the same for tile B
//   warp 8      TMA producer: Q_A, Q_B, then K_0, then (K_{j+1}, V_j) per tile
//   warp 9      TMEM allocator and MMA issuer (one thread)
//   warps 10-11 idle
// Per KV tile j the MMA warp issues S_A(j+1), S_B(j+1) as soon as each softmax
// warpgroup has copied S(j) to registers, then O^T += V_j^T P(j) once both
// warpgroups have written P(j).  A warpgroup writes P(j+1) only after
// O^T += V_j^T P(j) has completed (P has one buffer).
//
// Online softmax per row in log2 units (x = s * scale * log2 e), lazy
// rescale: the reference maximum moves only when a row's maximum grows by
// more than 8 (a factor 256); then that row's column of O^T and its sum are
// scaled by 2^(m_old - m_new).  Causal mask: score (i, j) = -inf for key
// j > query i, only in tiles that cross the diagonal ("Transformer"
// (ai-notes), section "What is the causal mask?").
//
// Boundaries between units: the producer prefetches the next unit's Q tiles
// into L2 when a unit starts; the next Q is rotated (RoPE) in shared memory as
// soon as it lands; when both tiles hold the same positions the two
// warpgroups split the channels and share the angles.  The epilogue
// normalises O^T by 1/l, transposes it into the warpgroup's rows of the P
// buffer (the layout of a 64-channel x 128-row swizzled TMA box) and stores
// it with two TMA tensor stores, which clip rows >= T.
#include "fwd_units.cuh"

namespace csattn {
namespace {

using namespace fwd;


constexpr int D = 128;                               // head size of v and out
constexpr int NS = 3;                                // K/V ring stages
constexpr int TILE_BYTES = BM * D * 2;              // 32 KB (a Q or K tile of d_k = 64 uses half)
constexpr int BLOCK_BYTES = BM * 128;               // 16 KB
constexpr int P_BYTES = 2 * BM * BN * 2;            // 64 KB: 256 rows x 128 keys
constexpr int SMEM_DATA = (2 + NS) * TILE_BYTES + P_BYTES;  // 229376
constexpr int SMEM_BYTES = SMEM_DATA + 512 + 1024;  // + barriers + per-query factors
constexpr uint32_t IDESC_PVT = idesc_bf16_f32(128, 256, 1, 0);  // A = V^T MN-major, B = P K-major

// byte offset of the 16-byte chunk holding keys [8c, 8c+8) of P row r
// (two 64-key column blocks of 256 rows x 128 bytes, 128-byte swizzle)
__device__ __forceinline__ uint32_t p_off(int r, int c) {
  return static_cast<uint32_t>((c >> 3) * (2 * BM * 128) + r * 128 + (((c & 7) ^ (r & 7)) << 4));
}

__device__ __forceinline__ void mbar_arrive_cnt(uint64_t* bar, uint32_t count) {
  asm volatile(
      "{\n\t.reg .b64 st;\n\t"
      "mbarrier.arrive.shared::cta.b64 st, [%0], %1;\n\t}" ::"r"(smem_u32(bar)),
      "r"(count)
      : "memory");
}

// TMA tiled store of one box from shared memory; completion tracked by bulk groups
__device__ __forceinline__ void tma_store_3d(const CUtensorMap* m, const void* smem_src, int x,
                                             int y, int z) {
  asm volatile(
      "cp.async.bulk.tensor.3d.global.shared::cta.bulk_group [%0, {%2, %3, %4}], [%1];" ::"l"(
          reinterpret_cast<uint64_t>(m)),
      "r"(smem_u32(smem_src)), "r"(x), "r"(y), "r"(z)
      : "memory");
}
__device__ __forceinline__ void bulk_commit() { asm volatile("cp.async.bulk.commit_group;" ::: "memory"); }
// the shared-memory source of every committed store has been read
__device__ __forceinline__ void bulk_wait_read() {
  asm volatile("cp.async.bulk.wait_group.read 0;" ::: "memory");
}
// every committed store has completed
__device__ __forceinline__ void bulk_wait_all() {
  asm volatile("cp.async.bulk.wait_group 0;" ::: "memory");
}

// L2 prefetch of one TMA box (no shared memory involved)
__device__ __forceinline__ void tma_prefetch_l2_3d(const CUtensorMap* m, int x, int y, int z) {
  asm volatile("cp.async.bulk.prefetch.tensor.3d.L2.global.tile [%0, {%1, %2, %3}];" ::"l"(
                   reinterpret_cast<uint64_t>(m)),
               "r"(x), "r"(y), "r"(z)
               : "memory");
}

// RoPE of 16-channel chunks [c_begin, c_end) of row r in one or two Q tiles (head size
// DK) at the same position: the angles are computed once and applied to both tiles.
template <int DK>
__device__ __forceinline__ void rotate_chunks(uint8_t* tile0, uint8_t* tile1, int r, int pos,
                                              int layout, const RopeTable& th, int c_begin,
                                              int c_end) {
#pragma unroll 2
  for (int c = c_begin; c < c_end; ++c) {
    int e0, e1;
    if (layout == 1) {
      e0 = 8 * c;
      e1 = DK / 2 + 8 * c;
    } else {
      e0 = 16 * c;
      e1 = 16 * c + 8;
    }
    float cs[8], sn[8];
#pragma unroll
    for (int i = 0; i < 8; ++i)
      rope_cos_sin<false>(pos, th.hi[8 * c + i], th.lo[8 * c + i], cs[i], sn[i]);
#pragma unroll
    for (int w = 0; w < 2; ++w) {
      uint8_t* tile = w ? tile1 : tile0;
      if (tile == nullptr) break;
      uint4* p0 = reinterpret_cast<uint4*>(tile + sw128_off(r, e0));
      uint4* p1 = reinterpret_cast<uint4*>(tile + sw128_off(r, e1));
      const uint4 a = *p0, b = *p1;
      const uint32_t wa[4] = {a.x, a.y, a.z, a.w};
      const uint32_t wb[4] = {b.x, b.y, b.z, b.w};
      float u[8], v[8];
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        u[2 * i] = bf16lo_to_f32(wa[i]);
        u[2 * i + 1] = bf16hi_to_f32(wa[i]);
        v[2 * i] = bf16lo_to_f32(wb[i]);
        v[2 * i + 1] = bf16hi_to_f32(wb[i]);
      }
      float ou[8], ov[8];
      if (layout == 1) {
#pragma unroll
        for (int i = 0; i < 8; ++i) {
          ou[i] = fmaf(u[i], cs[i], -v[i] * sn[i]);
          ov[i] = fmaf(u[i], sn[i], v[i] * cs[i]);
        }
      } else {
#pragma unroll
        for (int i = 0; i < 4; ++i) {
          ou[2 * i] = fmaf(u[2 * i], cs[i], -u[2 * i + 1] * sn[i]);
          ou[2 * i + 1] = fmaf(u[2 * i], sn[i], u[2 * i + 1] * cs[i]);
          ov[2 * i] = fmaf(v[2 * i], cs[4 + i], -v[2 * i + 1] * sn[4 + i]);
          ov[2 * i + 1] = fmaf(v[2 * i], sn[4 + i], v[2 * i + 1] * cs[4 + i]);
        }
      }
      *p0 = make_uint4(pack_bf16x2(ou[0], ou[1]), pack_bf16x2(ou[2], ou[3]),
                       pack_bf16x2(ou[4], ou[5]), pack_bf16x2(ou[6], ou[7]));
      *p1 = make_uint4(pack_bf16x2(ov[0], ov[1]), pack_bf16x2(ov[2], ov[3]),
                       pack_bf16x2(ov[4], ov[5]), pack_bf16x2(ov[6], ov[7]));
    }
  }
}

__device__ __forceinline__ void bar_sync_wg(int id) {
  asm volatile("bar.sync %0, 128;" ::"r"(id) : "memory");
}

// OR of `pred` over the 128 threads of a warpgroup (named barrier with reduction)
__device__ __forceinline__ bool bar_or_wg(int id, bool pred) {
  uint32_t r;
  asm volatile(
      "{\n\t.reg .pred p, q;\n\t"
      "setp.ne.u32 p, %1, 0;\n\t"
      "barrier.cta.red.or.pred q, %2, 128, p;\n\t"
      "selp.u32 %0, 1, 0, q;\n\t}"
      : "=r"(r)
      : "r"(pred ? 1u : 0u), "r"(id)
      : "memory");
  return r != 0;
}

// O^T += V^T P for 128 keys: eight MMAs, M=128 (d), N=256 (queries), K=16
template <bool LIMITED = false>
__device__ __forceinline__ void issue_pvt(uint32_t d_tmem, uint32_t v_smem, uint32_t p_smem,
                                          bool accumulate, int k_steps = BN / 16) {
#pragma unroll
  for (int kk = 0; kk < BN / 16; ++kk) {
    if (LIMITED && kk >= k_steps) break;
    const uint64_t a = smem_desc_sw128(v_smem + 2048u * kk, BM * 128, 1024);
    const uint64_t b = smem_desc_sw128(
        p_smem + static_cast<uint32_t>((kk >> 2) * (2 * BM * 128) + (kk & 3) * 32), 16, 1024);
    umma_ss(d_tmem, a, b, IDESC_PVT, (accumulate || kk > 0) ? 1u : 0u);
  }
}

// O^T += V^T P^T for a paged sequence's last key tile, whose rows past the end
// (nvalid..BN-1) may hold anything, NaN included, which P = 0 would not cancel:
// the 16-key steps past the end are skipped and the rows of the last step that lie
// past it are zeroed first.  Kept out of line so that the MMA thread's loop stays as
// compact as the contiguous kernel's (inlined, it cost the paged kernel 3 %).
__device__ __noinline__ void pvt_tail(uint32_t d_tmem, uint32_t v_smem, uint8_t* v_tile,
                                      uint32_t p_smem, bool accumulate, int nvalid) {
  const int k_steps = (nvalid + 15) / 16;
  for (int kb = 0; kb < D / 64; ++kb)
    for (int r = nvalid; r < 16 * k_steps; ++r)
      for (int c = 0; c < 8; ++c)
        *reinterpret_cast<uint4*>(v_tile + kb * BLOCK_BYTES + r * 128 + c * 16) =
            make_uint4(0u, 0u, 0u, 0u);
  fence_proxy_async_smem();
  issue_pvt<true>(d_tmem, v_smem, p_smem, accumulate, k_steps);
}

// DK: head size of q and k (64 or 128); v and out have D = 128 channels.
// PAGED: K/V from a paged cache with per-sequence lengths (see Params).
template <int DK, bool PAGED>
__global__ void __launch_bounds__(kThreads, 1)
    fwd_d128_kernel(const __grid_constant__ Params p, const __grid_constant__ CUtensorMap tm_q,
                    const __grid_constant__ CUtensorMap tm_k,
                    const __grid_constant__ CUtensorMap tm_v,
                    const __grid_constant__ CUtensorMap tm_o) {
  extern __shared__ __align__(1024) uint8_t smem[];
  uint8_t* sQ[2] = {smem, smem + TILE_BYTES};
  uint8_t* sKV = smem + 2 * TILE_BYTES;
  uint8_t* sP = smem + (2 + NS) * TILE_BYTES;
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + SMEM_DATA);
  uint64_t* q_full = bars + 0;
  uint64_t* q_ready = bars + 2;
  uint64_t* q_empty = bars + 4;
  uint64_t* s_full = bars + 6;
  uint64_t* s_free = bars + 8;
  uint64_t* p_full = bars + 10;   // one barrier, both warpgroups (8 warps)
  uint64_t* pv_done = bars + 11;  // O^T += V^T P(j) completed
  uint64_t* o_empty = bars + 12;  // epilogue of both tiles done (8 warps)
  uint64_t* teardown = bars + 13;
  uint64_t* kv_full = bars + 14;
  uint64_t* kv_empty = kv_full + NS;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(kv_empty + NS);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);
  volatile int* wg_fail = abort_flag + 1;                           // [2]
  float* rowf = reinterpret_cast<float*>(smem + SMEM_DATA + 512);  // [2][128]

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  if ((smem_u32(smem) & 1023u) != 0) {  // the swizzled layouts need a 1024-byte aligned base
    if (threadIdx.x == 0) atomicOr(p.status, kStatusDeviceArg);
    return;
  }

  if (threadIdx.x == 0) {
    for (int x = 0; x < 2; ++x) {
      mbar_init(&q_full[x], 1);
      mbar_init(&q_ready[x], 8);
      mbar_init(&q_empty[x], 1);
      mbar_init(&s_full[x], 1);
      mbar_init(&s_free[x], 4);
    }
    mbar_init(p_full, 8);
    mbar_init(pv_done, 1);
    mbar_init(o_empty, 8);
    mbar_init(teardown, 1);
    for (int s = 0; s < NS; ++s) {
      mbar_init(&kv_full[s], 1);
      mbar_init(&kv_empty[s], 1);
    }
    *abort_flag = 0;
    wg_fail[0] = 0;
    wg_fail[1] = 0;
    fence_mbar_init();
  }
  if (warp == kWarpMma) tmem_alloc(tmem_slot, 512);
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;

  if (warp >= 8) {
   regs_dec<kRegsCtl>();
   if (warp == kWarpProducer) {
    // ------------------------------------------------------------ TMA producer
    if (lane == 0) {
      tma_prefetch_desc(&tm_q);
      tma_prefetch_desc(&tm_k);
      tma_prefetch_desc(&tm_v);
      tma_prefetch_desc(&tm_o);
      uint32_t fill = 0;
      uint32_t nq[2] = {0, 0};
      bool ok = true;
      // one K (DK channels) or V (D channels) tile into the next ring stage
      auto load = [&](const CUtensorMap* m, int width, int j, const Unit& un) {
        const uint32_t s = fill % NS, use = fill / NS;
        if (use > 0 && !ctl_wait(&kv_empty[s], (use - 1) & 1, abort_flag, p.status, kWaitNs)) {
          ok = false;
          return;
        }
        mbar_arrive_expect_tx(&kv_full[s], static_cast<uint32_t>(BN * width * 2));
        uint8_t* dst = sKV + s * TILE_BYTES;
        if constexpr (!PAGED) {
          const int z = un.b * p.Hkv + un.kvh;
          for (int kb = 0; kb < width / 64; ++kb)
            tma_load_3d(dst + kb * BLOCK_BYTES, m, &kv_full[s], kb * 64, j * BN, z);
        } else {
          // paged: a box of box_rows rows never crosses a page; a box past the
          // sequence, or a page index outside the pool (reported), reads zeros (its
          // plane coordinate is past the tensor map)
          for (int r0 = 0; r0 < BN; r0 += p.box_rows) {
            const int t = j * BN + r0;
            int plane = p.num_pages * p.Hkv, prow = 0;
            if (t < un.Tk) {
              const int page = p.block_table[static_cast<size_t>(un.b) * p.max_pages +
                                             t / p.page_size];
              if (page >= 0 && page < p.num_pages)
                plane = page * p.Hkv + un.kvh;
              else
                atomicOr(p.status, kStatusDeviceArg);
              prow = t % p.page_size;
            }
            for (int kb = 0; kb < width / 64; ++kb)
              tma_load_3d(dst + kb * BLOCK_BYTES + r0 * 128, m, &kv_full[s], kb * 64, prow,
                          plane);
          }
        }
        ++fill;
      };
      for (int i = 0; ok; ++i) {
        const int u = unit_index(i);
        if (u >= p.nUnits) break;
        const Unit un = decode_unit<PAGED>(p, u);
        {
          // the next unit's Q tiles go to L2 now; their loads at the end of this unit hit it
          const int u2 = unit_index(i + 1);
          if (u2 < p.nUnits) {
            const Unit un2 = decode_unit<PAGED>(p, u2);
            for (int x = 0; x < 2; ++x)
              if (un2.n[x] > 0)
                for (int kb = 0; kb < DK / 64; ++kb)
                  tma_prefetch_l2_3d(&tm_q, kb * 64, un2.q0[x], un2.b * p.Hq + un2.h[x]);
          }
        }
#pragma unroll
        for (int x = 0; x < 2; ++x) {
          if (ok && un.n[x] > 0) {
            if (nq[x] > 0 &&
                !ctl_wait(&q_empty[x], (nq[x] - 1) & 1, abort_flag, p.status, kWaitNs)) {
              ok = false;
            } else {
              mbar_arrive_expect_tx(&q_full[x], static_cast<uint32_t>(BM * DK * 2));
#pragma unroll
              for (int kb = 0; kb < DK / 64; ++kb)
                tma_load_3d(sQ[x] + kb * BLOCK_BYTES, &tm_q, &q_full[x], kb * 64, un.q0[x],
                            un.b * p.Hq + un.h[x]);
              ++nq[x];
            }
          }
        }
        if (PAGED && un.bad_len) atomicOr(p.status, kStatusDeviceArg);
        // K leads V by one tile: K_0, then (K_{j+1}, V_j) for each j
        const int n = un.n[1];
        if (ok) load(&tm_k, DK, 0, un);
        for (int j = 0; j < n && ok; ++j) {
          if (j + 1 < n) load(&tm_k, DK, j + 1, un);
          if (ok) load(&tm_v, D, j, un);
        }
      }
      if (*abort_flag) {
        const uint32_t first = fill > static_cast<uint32_t>(NS) ? fill - NS : 0u;
        for (uint32_t f = first; f < fill; ++f)
          mbar_wait(&kv_full[f % NS], (f / NS) & 1, nullptr, p.status, kDrainNs);
        for (int x = 0; x < 2; ++x)
          if (nq[x] > 0) mbar_wait(&q_full[x], (nq[x] - 1) & 1, nullptr, p.status, kDrainNs);
      }
    }
   } else if (warp == kWarpMma) {
    // ------------------------------------------------------------ MMA issuer
    if (lane == 0) {
      const uint32_t sKV0 = smem_u32(sKV);
      const uint32_t sP0 = smem_u32(sP);
      const uint32_t sQa[2] = {smem_u32(sQ[0]), smem_u32(sQ[1])};
      const uint32_t tS[2] = {tmem + 0u, tmem + 128u};
      const uint32_t tO = tmem + 256u;
      uint32_t fill = 0, cq[2] = {0, 0}, cfree[2] = {0, 0}, cp = 0, units = 0;
      bool ok = true;
      auto wait = [&](uint64_t* bar, uint32_t parity) {
        if (!ok) return false;
        ok = ctl_wait(bar, parity, abort_flag, p.status, kWaitNs);
        tc_fence_after();
        return ok;
      };
      auto stage = [&](uint32_t f) { return sKV0 + (f % NS) * TILE_BYTES; };
      for (int i = 0; ok; ++i) {
        const int u = unit_index(i);
        if (u >= p.nUnits) break;
        const Unit un = decode_unit<PAGED>(p, u);
        const int n = un.n[1];
        // S(0) for both tiles (an absent tile A still runs: its rows are masked to P = 0)
        const uint32_t fK0 = fill++;
        if (!wait(&kv_full[fK0 % NS], (fK0 / NS) & 1)) break;
#pragma unroll
        for (int x = 0; x < 2; ++x) {
          if (un.n[x] > 0) {
            if (!wait(&q_ready[x], cq[x] & 1)) break;
            ++cq[x];
          }
          issue_qk<DK>(tS[x], sQa[x], stage(fK0));
          tc_commit(&s_full[x]);
          if (n == 1 && un.n[x] > 0) tc_commit(&q_empty[x]);
        }
        if (!ok) break;
        tc_commit(&kv_empty[fK0 % NS]);
        for (int j = 0; j < n && ok; ++j) {
          if (j + 1 < n) {
            const uint32_t fK = fill++;
            if (!wait(&kv_full[fK % NS], (fK / NS) & 1)) break;
#pragma unroll
            for (int x = 0; x < 2; ++x) {
              if (!wait(&s_free[x], cfree[x] & 1)) break;
              ++cfree[x];
              issue_qk<DK>(tS[x], sQa[x], stage(fK));
              tc_commit(&s_full[x]);
              if (j + 1 == n - 1 && un.n[x] > 0) tc_commit(&q_empty[x]);
            }
            if (!ok) break;
            tc_commit(&kv_empty[fK % NS]);
          } else {
            // the softmax warpgroups still release S(n-1); keep the count in step
#pragma unroll
            for (int x = 0; x < 2; ++x) {
              if (!wait(&s_free[x], cfree[x] & 1)) break;
              ++cfree[x];
            }
            if (!ok) break;
          }
          const uint32_t fV = fill++;
          if (!wait(&kv_full[fV % NS], (fV / NS) & 1)) break;
          if (!wait(p_full, cp & 1)) break;
          ++cp;
          if (j == 0 && units > 0 && !wait(o_empty, (units - 1) & 1)) break;
          if (PAGED && (j + 1) * BN > un.Tk)
            pvt_tail(tO, stage(fV), sKV + (fV % NS) * TILE_BYTES, sP0, j > 0, un.Tk - j * BN);
          else
            issue_pvt(tO, stage(fV), sP0, j > 0);
          tc_commit(pv_done);
          tc_commit(&kv_empty[fV % NS]);
        }
        ++units;
      }
      tc_commit(teardown);
      mbar_wait(teardown, 0, nullptr, p.status, kDrainNs);
    }
    __syncwarp();
   }
  } else {
    // ------------------------------------------------------------ softmax (A: warps 0-3, B: 4-7)
    // A failed wait never leaves the loops on its own: the warpgroup leaves together, after a
    // named-barrier reduction of the failure, so that no warp is left waiting at a named barrier.
    regs_inc<kRegsSoftmax>();
    const int x = warp >> 2;
    const int row = threadIdx.x & 127;               // query row of S = channel of O^T = TMEM lane
    const uint32_t lane_off = static_cast<uint32_t>((warp & 3) * 32) << 16;
    const uint32_t tS = tmem + lane_off + (x == 0 ? 0u : 128u);
    const uint32_t tOx = tmem + lane_off + 256u + static_cast<uint32_t>(x * BM);
    float* fct = rowf + x * BM;                      // per-query factors of this tile
    const float sl2 = p.scale_log2;
    const int bar_id = 1 + x;                        // named barrier of this warpgroup
    uint32_t cs = 0, cpv = 0;
    bool fail = false;
    // Wait for the next unit's Q and apply RoPE in shared memory.  When both tiles hold
    // the same positions (two heads of one KV group) each warpgroup rotates half of the
    // channels of both tiles, sharing the angles; otherwise it rotates its own tile.
    // q_ready completes after 8 warp arrivals either way.
    uint32_t cqa = 0, cqb = 0;  // Q tile loads seen per buffer
    auto prep_q = [&](int i_from) {
      for (int i2 = i_from;; ++i2) {
        const int u2 = unit_index(i2);
        if (u2 >= p.nUnits) return;
        const Unit un2 = decode_unit<PAGED>(p, u2);
        const bool shared_pos = un2.n[0] > 0 && un2.q0[0] == un2.q0[1];
        if (shared_pos) {
          if (fail || !warp_wait(&q_full[0], cqa & 1, abort_flag, p.status, kWaitNs) ||
              !warp_wait(&q_full[1], cqb & 1, abort_flag, p.status, kWaitNs)) {
            fail = true;
            return;
          }
          ++cqa;
          ++cqb;
          if (p.rope) {
            rotate_chunks<DK>(sQ[0], sQ[1], row, (PAGED ? un2.q_off : p.q_off) + un2.q0[0] + row, p.rope, p.theta,
                              x * (DK / 32), (x + 1) * (DK / 32));
            fence_proxy_async_smem();
          }
          __syncwarp();
          if (lane == 0) {
            mbar_arrive(&q_ready[0]);
            mbar_arrive(&q_ready[1]);
          }
          return;
        }
        // an absent tile (tile A of the last, single-tile pair) has nothing to rotate;
        // this warpgroup still runs that unit (masked) and prepares the next one after it
        if ((x ? un2.n[1] : un2.n[0]) == 0) return;
        uint32_t& cq = x ? cqb : cqa;
        if (fail || !warp_wait(&q_full[x], cq & 1, abort_flag, p.status, kWaitNs)) {
          fail = true;
          return;
        }
        ++cq;
        if (p.rope) {
          rotate_chunks<DK>(x ? sQ[1] : sQ[0], nullptr, row, (PAGED ? un2.q_off : p.q_off) + (x ? un2.q0[1] : un2.q0[0]) + row,
                        p.rope, p.theta,
                        0, DK / 16);
          fence_proxy_async_smem();
        }
        __syncwarp();
        if (lane == 0) mbar_arrive_cnt(&q_ready[x], 2);
        return;
      }
    };
    // true on every thread of the warpgroup when any of its warps has failed
    auto wg_failed = [&]() {
      if (fail) wg_fail[x] = 1;
      return bar_or_wg(bar_id, fail);
    };
    prep_q(0);
    for (int i = 0;; ++i) {
      const int u = unit_index(i);
      if (u >= p.nUnits) break;
      const Unit un = decode_unit<PAGED>(p, u);
      const int n = un.n[1];                       // both tiles step through tile B's keys
      const bool present = (x ? un.n[1] : un.n[0]) > 0;
      const int hx = x ? un.h[1] : un.h[0];
      const int qpos = (x ? un.q0[1] : un.q0[0]) + row;
      // paged: the last visible key of this row relative to tile 0, one register for the
      // whole unit (the causal bound and the sequence's end both shift by j * BN)
      const int lim0 = PAGED ? min(p.causal ? un.q_off + qpos : un.Tk - 1, un.Tk - 1) : 0;
      float m_used = -INFINITY, l = 0.f;
      bool leave = false;
      for (int j = 0; j < n; ++j) {
        if (!fail && !warp_wait(&s_full[x], cs & 1, abort_flag, p.status, kWaitNs)) fail = true;
        bool mine = false;
        float f = 1.0f;
        uint32_t pk[BN / 2];
        if (!fail) {
          ++cs;
          tc_fence_after();
          float s[BN];
          {
            uint32_t r[BN];
            tmem_ld128_sync(tS, r);
#pragma unroll
            for (int c = 0; c < BN; ++c) s[c] = __uint_as_float(r[c]);
          }
          // S(j) is in registers: the MMA warp may overwrite it with S(j+1)
          tc_fence_before();
          __syncwarp();
          if (lane == 0) mbar_arrive(&s_free[x]);
          int lim = BN - 1;
          if constexpr (PAGED) {
            lim = min(lim, lim0 - j * BN);
          } else {
            if (p.causal) lim = min(lim, p.q_off + qpos - j * BN);
            lim = min(lim, p.Tk - 1 - j * BN);
          }
          if (!present) lim = -1;
          if (lim < BN - 1) {
#pragma unroll
            for (int c = 0; c < BN; ++c) s[c] = (c <= lim) ? s[c] : -INFINITY;
          }
          float mq[4];
#pragma unroll
          for (int t = 0; t < 4; ++t) mq[t] = fmaxf(s[t], s[4 + t]);
#pragma unroll
          for (int c = 8; c < BN; c += 8) {
#pragma unroll
            for (int t = 0; t < 4; ++t) mq[t] = fmax3(mq[t], s[c + t], s[c + 4 + t]);
          }
          const float mx = fmaxf(fmaxf(mq[0], mq[1]), fmaxf(mq[2], mq[3]));
          const float m_new = fmaxf(m_used, mx * sl2);
          // lazy rescale: move the reference maximum only when it grew past the threshold
          mine = (j > 0) && (m_new > m_used + kRescaleThreshold);
          f = mine ? ex2_approx(m_used - m_new) : 1.0f;
          if (j == 0 || mine) m_used = m_new;
          const float neg_m = (m_used == -INFINITY) ? 0.f : -m_used;
          float sa0 = 0.f, sa1 = 0.f, sb0 = 0.f, sb1 = 0.f;
#pragma unroll
          for (int t = 0; t < BN / 2; ++t) {
            float x0, x1;
            ffma2(x0, x1, s[2 * t], s[2 * t + 1], sl2, sl2, neg_m, neg_m);
            const float p0 = ex2_approx(x0);
            const float p1 = ex2_approx(x1);
            if (t & 1)
              fadd2(sb0, sb1, sb0, sb1, p0, p1);
            else
              fadd2(sa0, sa1, sa0, sa1, p0, p1);
            pk[t] = pack_bf16x2(p0, p1);
          }
          l = l * f + ((sa0 + sa1) + (sb0 + sb1));
        }
        if (j > 0) {
          // the P buffer and O^T are free once O^T += V^T P(j-1) has completed
          if (!fail && !warp_wait(pv_done, cpv & 1, abort_flag, p.status, kWaitNs)) fail = true;
          if (!fail) {
            ++cpv;
            tc_fence_after();
          } else {
            wg_fail[x] = 1;
          }
          if (bar_or_wg(bar_id, mine || fail)) {
            fct[row] = f;
            bar_sync_wg(bar_id);
            const bool abort_wg = wg_fail[x] != 0;
            if (!abort_wg) {
              // this thread owns channel `row` of O^T: scale each query column by its factor
#pragma unroll 1
              for (int cb = 0; cb < BN; cb += 32) {
                uint32_t r[32];
                tmem_ld32_sync(tOx + static_cast<uint32_t>(cb), r);
#pragma unroll
                for (int c = 0; c < 32; c += 4) {
                  const float4 g = *reinterpret_cast<const float4*>(fct + cb + c);
                  r[c] = __float_as_uint(__uint_as_float(r[c]) * g.x);
                  r[c + 1] = __float_as_uint(__uint_as_float(r[c + 1]) * g.y);
                  r[c + 2] = __float_as_uint(__uint_as_float(r[c + 2]) * g.z);
                  r[c + 3] = __float_as_uint(__uint_as_float(r[c + 3]) * g.w);
                }
                tmem_st32(tOx + static_cast<uint32_t>(cb), r);
              }
              tmem_st_wait();
            }
            bar_sync_wg(bar_id);
            if (abort_wg) {
              fail = true;
              leave = true;
              break;
            }
          }
        }
        if (j == 0) {
          // the previous unit's output store reads these rows of the P buffer
          if (row == 0) bulk_wait_read();
          bar_sync_wg(bar_id);
        }
        if (!fail) {
          // P(j) row -> shared memory (K-major, swizzled), then hand it to the MMA warp
          const int pr = x * BM + row;
#pragma unroll
          for (int c = 0; c < BN / 8; ++c)
            *reinterpret_cast<uint4*>(sP + p_off(pr, c)) =
                make_uint4(pk[4 * c], pk[4 * c + 1], pk[4 * c + 2], pk[4 * c + 3]);
          fence_proxy_async_smem();
          tc_fence_before();
          __syncwarp();
          if (lane == 0) mbar_arrive(p_full);
        }
      }
      if (leave) break;
      prep_q(i + 1);
      // epilogue: wait for the last O^T += V^T P, normalise, transpose through this tile's
      // rows of the P buffer, store rows of out
      if (!fail && !warp_wait(pv_done, cpv & 1, abort_flag, p.status, kWaitNs)) fail = true;
      if (!fail) {
        ++cpv;
        tc_fence_after();
      }
      if (wg_failed()) break;
      fct[row] = l > 0.f ? 1.0f / l : 0.f;
      bar_sync_wg(bar_id);
      if (present) {
        // this thread holds channel `row` of O^T for the 128 queries of tile X: normalise
        // and write out[q][row] into this tile's rows of the P buffer, which then hold the
        // output tile in the layout of a 64-channel x 128-row swizzled TMA box per half
        uint8_t* const stg = sP + (row >> 6) * (2 * BM * 128) + x * (BM * 128) + ((row & 7) << 1);
        const int cg = (row >> 3) & 7;
#pragma unroll 1
        for (int h = 0; h < BM; h += 64) {
          uint32_t r[64];
          tmem_ld64_sync(tOx + static_cast<uint32_t>(h), r);
#pragma unroll
          for (int q = 0; q < 64; q += 4) {
            const float4 g = *reinterpret_cast<const float4*>(fct + h + q);
            const float gs[4] = {g.x, g.y, g.z, g.w};
#pragma unroll
            for (int t2 = 0; t2 < 4; ++t2) {
              const int qq = q + t2;  // (h + qq) % 8 == qq % 8
              *reinterpret_cast<__nv_bfloat16*>(stg + (h + qq) * 128 + ((cg ^ (qq & 7)) << 4)) =
                  __float2bfloat16_rn(__uint_as_float(r[qq]) * gs[t2]);
            }
          }
        }
        fence_proxy_async_smem();
      }
      tc_fence_before();
      bar_sync_wg(bar_id);
      if (present) {
        if (row == 0) {
          const int z = un.b * p.Hq + hx;
          const int q0x = x ? un.q0[1] : un.q0[0];
          tma_store_3d(&tm_o, sP + x * (BM * 128), 0, q0x, z);
          tma_store_3d(&tm_o, sP + 2 * BM * 128 + x * (BM * 128), 64, q0x, z);
          bulk_commit();
        }
        if (p.lse != nullptr && qpos < p.Tq)
          p.lse[(static_cast<size_t>(un.b) * p.Hq + hx) * p.Tq + qpos] =
              (m_used + log2f(l)) * 0.69314718055994531f;
      }
      __syncwarp();
      if (lane == 0) mbar_arrive(o_empty);
    }
    if (row == 0) bulk_wait_all();
  }

  tc_fence_before();
  __syncthreads();
  if (warp == kWarpMma) {
    tc_fence_after();
    tmem_dealloc(tmem, 512);
  }
}

template <int DK, bool PAGED>
cudaError_t launch_dk(const FwdArgs& a, const void* k_eff, cudaStream_t stream) {
  const Params p = make_params(a);
  alignas(64) CUtensorMap tq, tk, tv, to;
  // K/V tensor maps: [B*Hkv planes, Tk rows], or the page pool [num_pages*Hkv, page_size]
  const bool paged = a.block_table != nullptr;
  const int kv_rows = paged ? a.page_size : a.Tk;
  const int kv_planes = paged ? a.num_pages * a.Hkv : a.B * a.Hkv;
  if (!make_tmap_bf16_3d(&tq, a.q, DK, a.Tq, a.B * a.Hq, BM) ||
      !make_tmap_bf16_3d(&tk, k_eff, DK, kv_rows, kv_planes, p.box_rows) ||
      !make_tmap_bf16_3d(&tv, a.v, D, kv_rows, kv_planes, p.box_rows) ||
      !make_tmap_bf16_3d(&to, a.out, D, a.Tq, a.B * a.Hq, BM))
    return cudaErrorInvalidValue;
  static SmemLimitOnce smem_limit;
  cudaError_t e = smem_limit.set(fwd_d128_kernel<DK, PAGED>, SMEM_BYTES);
  if (e != cudaSuccess) return e;
  const int grid = p.nUnits < a.num_sms ? p.nUnits : a.num_sms;
  fwd_d128_kernel<DK, PAGED><<<grid, kThreads, SMEM_BYTES, stream>>>(p, tq, tk, tv, to);
  return cudaGetLastError();
}

}  // namespace

// v and out with 128 channels; q and k with a.d = 64 or 128
cudaError_t launch_fwd_sm103a_d128(const FwdArgs& a, const void* k_eff, cudaStream_t stream) {
  if (a.block_table != nullptr)
    return a.d == 128 ? launch_dk<128, true>(a, k_eff, stream) : cudaErrorInvalidValue;
  if (a.d == 128) return launch_dk<128, false>(a, k_eff, stream);
  if (a.d == 64) return launch_dk<64, false>(a, k_eff, stream);
  return cudaErrorInvalidValue;
}

}  // namespace csattn
