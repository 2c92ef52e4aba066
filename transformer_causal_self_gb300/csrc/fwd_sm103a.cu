// Causal GQA attention prefill for head size 64, bf16 in / bf16 out, fp32
// accumulation, for sm_103a: TMA tiles into shared memory, tcgen05 MMAs with
// TMEM accumulators, online softmax in fp32.  The T x T score matrix never
// leaves the SM ("Grasping Codes and Math 02", section "Flash Attention: The
// GPU Does Everything in One Pass": same result without materialising the
// matrix).  Head size 128 runs the kernel in fwd_sm103a_d128.cu; the unit
// schedule and shared helpers are in fwd_units.cuh.
//
// Warp roles (384 threads = three warpgroups; setmaxnreg gives the softmax
// warpgroups 200 registers and the third 104: 2*128*200 + 128*104 = 384*168):
//   warps 0-3   softmax for tile A (TMEM lanes 0-127 = query rows); also the
//               RoPE of tile A's next Q and tile A's epilogue
//   warps 4-7   the same for tile B
//   warp 8      TMA producer: Q_A, Q_B, then K_0, V_0, K_1, V_1, ... into a ring
//   warp 9      TMEM allocator and MMA issuer (one thread)
//   warps 10-11 idle (they complete the third warpgroup)
// At the end of a unit a softmax warpgroup rotates the next unit's Q (which
// has landed by then) before its epilogue, so the MMA warp can start the next
// unit's S = Q K^T while the epilogue stores O.
// TMEM columns: S_A [0,128) S_B [128,256) O_A [256,256+D) O_B [256+D,256+2D), with D
// the head size of v and out (64); q and k have DK = 64 or 128 channels.
// P (bf16) overwrites the first 64 columns of its S region and feeds the
// second MMA straight from TMEM.
//
// MMA order per KV tile j (per unit):  PV_A(j) S_A(j+1) PV_B(j) S_B(j+1), so
// each softmax warpgroup has two MMAs' time to turn S(j+1) into P(j+1) while
// the tensor core works on the other tile.
//
// Online softmax per row (scores in log2 units, x = s * scale * log2 e):
//   m = running max used for the exponent, l = running sum, O in TMEM.
//   A new tile raises m only when its max exceeds m by more than 8 (a factor
//   256); then O and l are rescaled by 2^(m_old - m_new).  P = 2^(x - m) <= 256.
// Causal mask: score (i, j) = -inf when key j > query i, applied only in the
// tiles that cross the diagonal; tiles entirely above it are skipped
// ("Transformer" (ai-notes), section "What is the causal mask?").
#include "fwd_units.cuh"

namespace csattn {
namespace {

using namespace fwd;

template <int DK, int D>
struct Cfg {
  static constexpr int BLOCK_BYTES = BM * 128;   // one column block of a 128-row tile
  static constexpr int Q_BYTES = BM * DK * 2;    // one Q or K tile
  static constexpr int V_BYTES = BM * D * 2;     // one V tile
  static constexpr int TILE_BYTES = Q_BYTES > V_BYTES ? Q_BYTES : V_BYTES;  // a ring stage
  static constexpr int NS = DK == 64 ? 8 : 4;    // K/V ring stages
  static constexpr int SMEM_TILE_BYTES = 2 * Q_BYTES + NS * TILE_BYTES;
  static constexpr int SMEM_BYTES = SMEM_TILE_BYTES + 1024 + 1024;
  static constexpr uint32_t TMEM_COLS = 512;
  static constexpr uint32_t IDESC_PV = idesc_bf16_f32(128, D, 0, 1);
};

// O (+)= P V: M=128, N=D, K=128 keys; P from TMEM, V MN-major (rows = keys).
// LIMITED: only the first k_steps 16-key steps.
template <int DK, int D, bool LIMITED = false>
__device__ __forceinline__ void issue_pv(uint32_t d_tmem, uint32_t p_tmem, uint32_t v_smem,
                                         bool accumulate, int k_steps = BN / 16) {
#pragma unroll
  for (int kk = 0; kk < BN / 16; ++kk) {
    if (LIMITED && kk >= k_steps) break;
    umma_ts(d_tmem, p_tmem + 8u * kk, smem_desc_sw128(v_smem + 2048u * kk, BM * 128, 1024),
            Cfg<DK, D>::IDESC_PV, (accumulate || kk > 0) ? 1u : 0u);
  }
}

// A paged sequence's last key tile (paged kernel only): its rows past the end
// (nvalid..BN-1) may hold anything, NaN included, which P = 0 would not cancel.  The
// rows of the last 16-key step that lie past the end are zeroed here (the steps after
// it are not issued), out of line so that the MMA thread's loop stays compact.
template <int D>
__device__ __noinline__ void v_tail_zero(uint8_t* v_tile, int nvalid) {
  const int end = 16 * ((nvalid + 15) / 16);
  for (int kb = 0; kb < D / 64; ++kb)
    for (int r = nvalid; r < end; ++r)
      for (int c = 0; c < 8; ++c)
        *reinterpret_cast<uint4*>(v_tile + kb * BM * 128 + r * 128 + c * 16) =
            make_uint4(0u, 0u, 0u, 0u);
  fence_proxy_async_smem();
}
template <int DK, int D>
__device__ __noinline__ void pv_tail(uint32_t d_tmem, uint32_t p_tmem, uint32_t v_smem,
                                     bool accumulate, int nvalid) {
  issue_pv<DK, D, true>(d_tmem, p_tmem, v_smem, accumulate, (nvalid + 15) / 16);
}

// PAGED: K/V from a paged cache with per-sequence lengths (Params in fwd_units.cuh).
template <int DK, int D, bool PAGED>
__global__ void __launch_bounds__(kThreads, 1)
    fwd_sm103a_kernel(const __grid_constant__ Params p, const __grid_constant__ CUtensorMap tm_q,
                      const __grid_constant__ CUtensorMap tm_k,
                      const __grid_constant__ CUtensorMap tm_v) {
  using C = Cfg<DK, D>;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~static_cast<uintptr_t>(1023));
  uint8_t* sQ[2] = {smem, smem + C::Q_BYTES};
  uint8_t* sKV = smem + 2 * C::Q_BYTES;
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + C::SMEM_TILE_BYTES);
  uint64_t* q_full = bars + 0;
  uint64_t* q_ready = bars + 2;
  uint64_t* q_empty = bars + 4;
  uint64_t* s_full = bars + 6;
  uint64_t* p_full = bars + 8;
  uint64_t* o_full = bars + 10;
  uint64_t* o_empty = bars + 12;
  uint64_t* teardown = bars + 14;
  uint64_t* kv_full = bars + 16;
  uint64_t* kv_empty = kv_full + C::NS;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(kv_empty + C::NS);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;

  if (threadIdx.x == 0) {
    for (int x = 0; x < 2; ++x) {
      mbar_init(&q_full[x], 1);
      mbar_init(&q_ready[x], 4);
      mbar_init(&q_empty[x], 1);
      mbar_init(&s_full[x], 1);
      mbar_init(&p_full[x], 4);
      mbar_init(&o_full[x], 1);
      mbar_init(&o_empty[x], 4);
    }
    mbar_init(teardown, 1);
    for (int s = 0; s < C::NS; ++s) {
      mbar_init(&kv_full[s], 1);
      mbar_init(&kv_empty[s], 1);
    }
    *abort_flag = 0;
    fence_mbar_init();
  }
  if (warp == kWarpMma) tmem_alloc(tmem_slot, C::TMEM_COLS);
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
      uint32_t fill = 0;
      uint32_t nq[2] = {0, 0};
      bool ok = true;
      for (int i = 0; ok; ++i) {
        const int u = unit_index(i);
        if (u >= p.nUnits) break;
        const Unit un = decode_unit<PAGED>(p, u);
#pragma unroll
        for (int x = 0; x < 2; ++x) {
          if (ok && un.n[x] > 0) {
            if (nq[x] > 0 &&
                !ctl_wait(&q_empty[x], (nq[x] - 1) & 1, abort_flag, p.status, kWaitNs)) {
              ok = false;
            } else {
              mbar_arrive_expect_tx(&q_full[x], C::Q_BYTES);
#pragma unroll
              for (int kb = 0; kb < DK / 64; ++kb)
                tma_load_3d(sQ[x] + kb * C::BLOCK_BYTES, &tm_q, &q_full[x], kb * 64, un.q0[x],
                            un.b * p.Hq + un.h[x]);
              ++nq[x];
            }
          }
        }
        if (PAGED && un.bad_len) atomicOr(p.status, kStatusDeviceArg);
        for (int j = 0; j < un.n[1] && ok; ++j) {
          for (int t = 0; t < 2; ++t) {
            const uint32_t s = fill % C::NS, use = fill / C::NS;
            if (use > 0 && !ctl_wait(&kv_empty[s], (use - 1) & 1, abort_flag, p.status, kWaitNs)) {
              ok = false;
              break;
            }
            mbar_arrive_expect_tx(&kv_full[s], t == 0 ? C::Q_BYTES : C::V_BYTES);
            uint8_t* dst = sKV + s * C::TILE_BYTES;
            if constexpr (!PAGED) {
              for (int kb = 0; kb < (t == 0 ? DK : D) / 64; ++kb)
                tma_load_3d(dst + kb * C::BLOCK_BYTES, t == 0 ? &tm_k : &tm_v, &kv_full[s],
                            kb * 64, j * BN, un.b * p.Hkv + un.kvh);
            } else {
              // paged: a box of box_rows rows never crosses a page; a box past the
              // sequence, or a page index outside the pool (reported), reads zeros
              for (int r0 = 0; r0 < BN; r0 += p.box_rows) {
                const int tr = j * BN + r0;
                int plane = p.num_pages * p.Hkv, prow = 0;
                if (tr < un.Tk) {
                  const int page = p.block_table[static_cast<size_t>(un.b) * p.max_pages +
                                                 tr / p.page_size];
                  if (page >= 0 && page < p.num_pages)
                    plane = page * p.Hkv + un.kvh;
                  else
                    atomicOr(p.status, kStatusDeviceArg);
                  prow = tr % p.page_size;
                }
                for (int kb = 0; kb < (t == 0 ? DK : D) / 64; ++kb)
                  tma_load_3d(dst + kb * C::BLOCK_BYTES + r0 * 128, t == 0 ? &tm_k : &tm_v,
                              &kv_full[s], kb * 64, prow, plane);
              }
            }
            ++fill;
          }
        }
      }
      if (*abort_flag) {
        // Let every copy still in flight land before the CTA's shared memory is released.
        const uint32_t first = fill > static_cast<uint32_t>(C::NS) ? fill - C::NS : 0u;
        for (uint32_t f = first; f < fill; ++f)
          mbar_wait(&kv_full[f % C::NS], (f / C::NS) & 1, nullptr, p.status, kDrainNs);
        for (int x = 0; x < 2; ++x)
          if (nq[x] > 0) mbar_wait(&q_full[x], (nq[x] - 1) & 1, nullptr, p.status, kDrainNs);
      }
    }
  } else if (warp == kWarpMma) {
    // ------------------------------------------------------------ MMA issuer
    if (lane == 0) {
      const uint32_t sKV0 = smem_u32(sKV);
      const uint32_t sQa[2] = {smem_u32(sQ[0]), smem_u32(sQ[1])};
      const uint32_t tS[2] = {tmem + 0u, tmem + 128u};
      const uint32_t tO[2] = {tmem + 256u, tmem + 256u + static_cast<uint32_t>(D)};
      uint32_t fill = 0;
      uint32_t cq[2] = {0, 0}, cp[2] = {0, 0}, cu[2] = {0, 0};
      bool ok = true;
      auto wait = [&](uint64_t* bar, uint32_t parity) {
        if (!ok) return false;
        ok = ctl_wait(bar, parity, abort_flag, p.status, kWaitNs);
        tc_fence_after();
        return ok;
      };
      for (int i = 0; ok; ++i) {
        const int u = unit_index(i);
        if (u >= p.nUnits) break;
        const Unit un = decode_unit<PAGED>(p, u);
        // first score tiles: S_X(0) = Q_X K_0^T
        const uint32_t s0 = fill % C::NS;
        bool k0_ready = false;
#pragma unroll
        for (int x = 0; x < 2; ++x) {
          if (un.n[x] > 0 && wait(&q_ready[x], cq[x] & 1)) {
            ++cq[x];
            if (!k0_ready) k0_ready = wait(&kv_full[s0], (fill / C::NS) & 1);
            if (k0_ready) {
              issue_qk<DK>(tS[x], sQa[x], sKV0 + s0 * C::TILE_BYTES);
              tc_commit(&s_full[x]);
              if (un.n[x] == 1) tc_commit(&q_empty[x]);
            }
          }
        }
        if (!ok) break;
        tc_commit(&kv_empty[s0]);
        for (int j = 0; j < un.n[1] && ok; ++j) {
          const uint32_t fV = fill + 2 * j + 1, fK = fill + 2 * j + 2;
          const uint32_t sV = fV % C::NS, sK = fK % C::NS;
          bool v_ready = false, k_ready = false;
#pragma unroll
          for (int x = 0; x < 2; ++x) {
            if (j < un.n[x] && wait(&p_full[x], cp[x] & 1)) {
              ++cp[x];
              const bool tail = PAGED && (j + 1) * BN > un.Tk;
              if (!v_ready) {
                v_ready = wait(&kv_full[sV], (fV / C::NS) & 1);
                if (tail && v_ready) v_tail_zero<D>(sKV + sV * C::TILE_BYTES, un.Tk - j * BN);
              }
              if (v_ready && (j > 0 || cu[x] == 0 || wait(&o_empty[x], (cu[x] - 1) & 1))) {
                if (tail)
                  pv_tail<DK, D>(tO[x], tS[x], sKV0 + sV * C::TILE_BYTES, j > 0, un.Tk - j * BN);
                else
                  issue_pv<DK, D>(tO[x], tS[x], sKV0 + sV * C::TILE_BYTES, j > 0);
                if (x == 1) tc_commit(&kv_empty[sV]);
                if (j == un.n[x] - 1) tc_commit(&o_full[x]);
                if (j + 1 < un.n[x]) {
                  if (!k_ready) k_ready = wait(&kv_full[sK], (fK / C::NS) & 1);
                  if (k_ready) {
                    issue_qk<DK>(tS[x], sQa[x], sKV0 + sK * C::TILE_BYTES);
                    tc_commit(&s_full[x]);
                    if (j + 1 == un.n[x] - 1) tc_commit(&q_empty[x]);
                    if (x == 1) tc_commit(&kv_empty[sK]);
                  }
                }
              }
            }
          }
        }
#pragma unroll
        for (int x = 0; x < 2; ++x)
          if (un.n[x] > 0) ++cu[x];
        fill += 2 * un.n[1];
      }
      // every MMA issued above has completed once this barrier flips
      tc_commit(teardown);
      mbar_wait(teardown, 0, nullptr, p.status, kDrainNs);
    }
    __syncwarp();
   }
  } else {
    // ------------------------------------------------------------ softmax (A: warps 0-3, B: 4-7)
    regs_inc<kRegsSoftmax>();
    const int x = warp >> 2;
    const int row = threadIdx.x & 127;
    const uint32_t lane_off = static_cast<uint32_t>((warp & 3) * 32) << 16;
    const uint32_t tS = tmem + lane_off + (x == 0 ? 0u : 128u);
    const uint32_t tO = tmem + lane_off + 256u + (x == 0 ? 0u : static_cast<uint32_t>(D));
    const float sl2 = p.scale_log2;
    uint32_t cq = 0, cs = 0, co = 0;
    bool ok = true;
    // Q of the next unit this warpgroup serves: wait for the tile, rotate row
    // `row`, hand it to the MMA warp.  Done right after a unit's last P and
    // before its epilogue, so the MMA warp can start the next unit's first
    // S = Q K^T while the epilogue runs.
    auto prep_q = [&](int i_from) {
      for (int i2 = i_from;; ++i2) {
        const int u2 = unit_index(i2);
        if (u2 >= p.nUnits) return;
        const Unit un2 = decode_unit<PAGED>(p, u2);
        if ((x ? un2.n[1] : un2.n[0]) == 0) continue;
        if (!warp_wait(&q_full[x], cq & 1, abort_flag, p.status, kWaitNs)) {
          ok = false;
          return;
        }
        ++cq;
        if (p.rope) {
          rotate_q_row<DK>(x ? sQ[1] : sQ[0], row,
                           (PAGED ? un2.q_off : p.q_off) + (x ? un2.q0[1] : un2.q0[0]) + row, p.rope,
                          p.theta);
          fence_proxy_async_smem();
        }
        __syncwarp();
        if (lane == 0) mbar_arrive(&q_ready[x]);
        return;
      }
    };
    prep_q(0);
    for (int i = 0; ok; ++i) {
      const int u = unit_index(i);
      if (u >= p.nUnits) break;
      const Unit un = decode_unit<PAGED>(p, u);
      const int n = x ? un.n[1] : un.n[0];
      if (n == 0) continue;
      const int hx = x ? un.h[1] : un.h[0];
      const int qpos = (x ? un.q0[1] : un.q0[0]) + row;
      // paged: the last visible key of this row relative to tile 0 (one register)
      const int lim0 = PAGED ? min(p.causal ? un.q_off + qpos : un.Tk - 1, un.Tk - 1) : 0;

      float m_used = -INFINITY, l = 0.f;
      for (int j = 0; j < n; ++j) {
        if (!warp_wait(&s_full[x], cs & 1, abort_flag, p.status, kWaitNs)) {
          ok = false;
          break;
        }
        ++cs;
        tc_fence_after();
        float s[BN];
        {
          uint32_t r[BN];
          tmem_ld128_sync(tS, r);
#pragma unroll
          for (int c = 0; c < BN; ++c) s[c] = __uint_as_float(r[c]);
        }
        // causal diagonal and ragged tail: keys beyond the row's limit get -inf
        int lim = BN - 1;
        if constexpr (PAGED) {
          lim = min(lim, lim0 - j * BN);
        } else {
          if (p.causal) lim = min(lim, p.q_off + qpos - j * BN);
          lim = min(lim, p.Tk - 1 - j * BN);
        }
        if (lim < BN - 1) {
#pragma unroll
          for (int c = 0; c < BN; ++c) s[c] = (c <= lim) ? s[c] : -INFINITY;
        }
        // row max as four independent chains (latency), then combined
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
        if (j == 0) {
          m_used = m_new;
        } else {
          const bool mine = m_new > m_used + kRescaleThreshold;
          if (__any_sync(0xffffffffu, mine)) {
            const float f = mine ? ex2_approx(m_used - m_new) : 1.0f;
            l *= f;
#pragma unroll 1
            for (int c = 0; c < D / 32; ++c) {
              uint32_t r[32];
              tmem_ld32_sync(tO + 32u * c, r);
#pragma unroll
              for (int t = 0; t < 32; ++t) r[t] = __float_as_uint(__uint_as_float(r[t]) * f);
              tmem_st32(tO + 32u * c, r);
            }
            tmem_st_wait();
            if (mine) m_used = m_new;
          }
        }
        float sa0 = 0.f, sa1 = 0.f, sb0 = 0.f, sb1 = 0.f;  // two independent pair sums
        const float neg_m = -m_used;
#pragma unroll
        for (int c = 0; c < BN / 64; ++c) {
          uint32_t pk[32];
#pragma unroll
          for (int t = 0; t < 32; ++t) {
            float x0, x1;
            ffma2(x0, x1, s[64 * c + 2 * t], s[64 * c + 2 * t + 1], sl2, sl2, neg_m, neg_m);
            const float p0 = ex2_approx(x0);
            const float p1 = ex2_approx(x1);
            if (t & 1)
              fadd2(sb0, sb1, sb0, sb1, p0, p1);
            else
              fadd2(sa0, sa1, sa0, sa1, p0, p1);
            pk[t] = pack_bf16x2(p0, p1);
          }
          tmem_st32(tS + 32u * c, pk);
        }
        l += (sa0 + sa1) + (sb0 + sb1);
        tmem_st_wait();
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(&p_full[x]);
      }
      if (!ok) break;
      prep_q(i + 1);
      if (!ok) break;
      // epilogue: O / l -> bf16 rows of out; optional natural-log LSE
      if (!warp_wait(&o_full[x], co & 1, abort_flag, p.status, kWaitNs)) break;
      ++co;
      tc_fence_after();
      const float inv = 1.f / l;
      const bool live = qpos < p.Tq;
      __nv_bfloat16* orow =
          p.out + ((static_cast<size_t>(un.b) * p.Hq + hx) * p.Tq + (live ? qpos : 0)) * D;
#pragma unroll 1
      for (int c = 0; c < D / 32; ++c) {
        uint32_t r[32];
        tmem_ld32_sync(tO + 32u * c, r);
        uint32_t w[16];
#pragma unroll
        for (int t = 0; t < 16; ++t)
          w[t] = pack_bf16x2(__uint_as_float(r[2 * t]) * inv, __uint_as_float(r[2 * t + 1]) * inv);
        if (live) {
          uint4* dst = reinterpret_cast<uint4*>(orow + 32 * c);
#pragma unroll
          for (int t = 0; t < 4; ++t) dst[t] = make_uint4(w[4 * t], w[4 * t + 1], w[4 * t + 2], w[4 * t + 3]);
        }
      }
      if (live && p.lse != nullptr)
        p.lse[(static_cast<size_t>(un.b) * p.Hq + hx) * p.Tq + qpos] =
            (m_used + log2f(l)) * 0.69314718055994531f;
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(&o_empty[x]);
    }
  }

  tc_fence_before();
  __syncthreads();
  if (warp == kWarpMma) {
    tc_fence_after();
    tmem_dealloc(tmem, C::TMEM_COLS);
  }
}

template <int DK, bool PAGED>
cudaError_t launch_v64(const FwdArgs& a, const void* k_eff, cudaStream_t stream) {
  constexpr int D = 64;
  using C = Cfg<DK, D>;
  const Params p = make_params(a);
  alignas(64) CUtensorMap tq, tk, tv;
  // K/V tensor maps: [B*Hkv planes, Tk rows], or the page pool [num_pages*Hkv, page_size]
  const int kv_rows = PAGED ? a.page_size : a.Tk;
  const int kv_planes = PAGED ? a.num_pages * a.Hkv : a.B * a.Hkv;
  if (!make_tmap_bf16_3d(&tq, a.q, DK, a.Tq, a.B * a.Hq, BM) ||
      !make_tmap_bf16_3d(&tk, k_eff, DK, kv_rows, kv_planes, p.box_rows) ||
      !make_tmap_bf16_3d(&tv, a.v, D, kv_rows, kv_planes, p.box_rows))
    return cudaErrorInvalidValue;
  static SmemLimitOnce smem_limit;
  cudaError_t e = smem_limit.set(fwd_sm103a_kernel<DK, D, PAGED>, C::SMEM_BYTES);
  if (e != cudaSuccess) return e;
  const int grid = p.nUnits < a.num_sms ? p.nUnits : a.num_sms;
  fwd_sm103a_kernel<DK, D, PAGED><<<grid, kThreads, C::SMEM_BYTES, stream>>>(p, tq, tk, tv);
  return cudaGetLastError();
}

}  // namespace

// q, k with a.d channels and v, out with a.dv channels, each 64 or 128: v of 128
// channels runs the O^T kernel (fwd_sm103a_d128.cu), v of 64 this file's kernel
cudaError_t launch_fwd_sm103a(const FwdArgs& a, const void* k_eff, cudaStream_t stream) {
  if (a.dv == 128) return launch_fwd_sm103a_d128(a, k_eff, stream);
  if (a.dv != 64) return cudaErrorInvalidValue;
  if (a.block_table != nullptr)
    return a.d == 64 ? launch_v64<64, true>(a, k_eff, stream) : cudaErrorInvalidValue;
  if (a.d == 64) return launch_v64<64, false>(a, k_eff, stream);
  if (a.d == 128) return launch_v64<128, false>(a, k_eff, stream);
  return cudaErrorInvalidValue;
}

}  // namespace csattn
