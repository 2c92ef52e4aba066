// Shared pieces of the two sm_103a prefill kernels (fwd_sm103a.cu for d = 64,
// fwd_sm103a_d128.cu for d = 128): constants, the kernel parameter block, the
// work-unit schedule, RoPE of a Q row in shared memory and the S = Q K^T MMA.
//
// Work unit: two 128-row query tiles (A and B) that read the same KV head.
// With a GQA group of >= 2 query heads, A and B are the same rows of two heads
// of the group, so every K/V tile is loaded once for both; otherwise they are
// two consecutive tiles of one head.  The CTA is persistent (one per SM) and
// walks the units longest-first in a snake order.
#pragma once
#include "internal.h"

namespace csattn {
namespace fwd {

constexpr int BM = 128;  // query rows per tile = TMEM lanes
constexpr int BN = 128;  // keys per KV tile
constexpr int kThreads = 384;
constexpr int kWarpProducer = 8;
constexpr int kWarpMma = 9;
constexpr int kRegsSoftmax = 200;  // 2*128*200 + 128*104 = 64512 = 384 * 168
constexpr int kRegsCtl = 104;
constexpr uint64_t kWaitNs = 2000000000ull;     // 2 s: far above any legal wait
constexpr uint64_t kDrainNs = 100000000ull;     // 100 ms for the teardown after an abort
constexpr float kRescaleThreshold = 8.0f;        // log2 units

constexpr uint32_t kIdescS = idesc_bf16_f32(128, 128, 0, 0);  // S = Q K^T, both K-major

struct Params {
  __nv_bfloat16* out;
  float* lse;
  uint32_t* status;
  int B, Hq, Hkv;
  int Tq, Tk;   // query rows, key rows
  int q_off;    // position of query row 0; keys sit at 0..Tk-1
  int rep;      // Hq / Hkv
  int hp;       // head pairs per group (rep / 2)
  int n_qt;     // ceil(Tq / 128) query tiles
  int n_kt;     // ceil(Tk / 128) key tiles
  int causal;   // key j visible to query row i iff j <= q_off + i
  int rope;     // 0 none, 1 split-half, 2 adjacent
  int nP;       // units made of head pairs
  int nUnits;   // all units
  float scale_log2;
  RopeTable theta;
  // Paged KV cache (the kernels' paged instances; block_table == nullptr otherwise): keys and
  // values of sequence b at rows 0..L_b+Tq-1 with L_b = cache_lens[b] (the cached
  // prefix, then the chunk's own rows); row t lives in page block_table[b * max_pages
  // + t / page_size] at offset t % page_size; K/V tensor maps span the page pool
  // with planes page * Hkv + kv head.  Query row i of sequence b sits at L_b + i.
  const int32_t* cache_lens;
  const int32_t* block_table;
  int page_size, num_pages, max_pages;
  int box_rows;  // rows per K/V TMA box: 128, 64, or the page size (16, 32)
};

struct Unit {
  int b, kvh;
  int h[2], q0[2], n[2];  // per tile: head, first row, number of key tiles (n[0] <= n[1])
  int q_off, Tk;          // position of query row 0 and key rows of this sequence
  bool bad_len;           // paged: cache_lens[b] out of range (run as L_b = 0, reported)
};

// Key tiles query tile qt reads: all of them, or (causal) up to the tile that holds
// the position of its last row.  Never 0 (key 0 is visible to every query).
__device__ __forceinline__ int key_tiles(const Params& p, int qt, int q_off, int n_kt) {
  if (!p.causal) return n_kt;
  const int last = min(qt * BM + BM, p.Tq) - 1 + q_off;
  return min(n_kt, last / BN + 1);
}

// Position of query row 0 and key count of sequence b: the call's, or from the
// paged cache's lengths (a length outside [0, max_pages * page_size - Tq] runs as 0).
template <bool PAGED>
__device__ __forceinline__ void seq_extent(const Params& p, Unit& r) {
  r.q_off = p.q_off;
  r.Tk = p.Tk;
  r.bad_len = false;
  if constexpr (PAGED) {
    int L = p.cache_lens[r.b];
    if (L < 0 || L > p.max_pages * p.page_size - p.Tq) {
      r.bad_len = true;
      L = 0;
    }
    r.q_off = L;
    r.Tk = L + p.Tq;
  }
}

// PAGED: per-sequence extents from the paged cache's lengths; otherwise the call's.
template <bool PAGED = false>
__device__ __forceinline__ Unit decode_unit(const Params& p, int u) {
  Unit r;
  if (u < p.nP) {
    const int per = p.B * p.Hkv * p.hp;
    int qt = u / per;
    int rem = u - qt * per;
    if (p.causal) qt = p.n_qt - 1 - qt;
    r.b = rem / (p.Hkv * p.hp);
    rem -= r.b * (p.Hkv * p.hp);
    r.kvh = rem / p.hp;
    const int pp = rem - r.kvh * p.hp;
    r.h[0] = r.kvh * p.rep + 2 * pp;
    r.h[1] = r.h[0] + 1;
    r.q0[0] = r.q0[1] = qt * BM;
    seq_extent<PAGED>(p, r);
    r.n[0] = r.n[1] = key_tiles(p, qt, r.q_off, PAGED ? (r.Tk + BN - 1) / BN : p.n_kt);
  } else {
    const int u2 = u - p.nP;
    const int npairs = (p.n_qt + 1) / 2;
    const int per = p.B * p.Hkv;
    int m = u2 / per;
    const int rem = u2 - m * per;
    if (p.causal) m = npairs - 1 - m;
    r.b = rem / p.Hkv;
    r.kvh = rem - r.b * p.Hkv;
    r.h[0] = r.h[1] = r.kvh * p.rep + p.rep - 1;
    seq_extent<PAGED>(p, r);
    const int t0 = 2 * m, t1 = 2 * m + 1;
    if (t1 < p.n_qt) {
      r.q0[0] = t0 * BM;
      r.n[0] = key_tiles(p, t0, r.q_off, PAGED ? (r.Tk + BN - 1) / BN : p.n_kt);
      r.q0[1] = t1 * BM;
      r.n[1] = key_tiles(p, t1, r.q_off, PAGED ? (r.Tk + BN - 1) / BN : p.n_kt);
    } else {
      r.q0[0] = 0;
      r.n[0] = 0;
      r.q0[1] = t0 * BM;
      r.n[1] = key_tiles(p, t0, r.q_off, PAGED ? (r.Tk + BN - 1) / BN : p.n_kt);
    }
  }
  return r;
}

__device__ __forceinline__ bool warp_wait(uint64_t* bar, uint32_t parity, volatile int* abort,
                                          uint32_t* status, uint64_t limit_ns) {
  const bool ok = mbar_wait(bar, parity, abort, status, limit_ns);
  return __all_sync(0xffffffffu, ok) != 0;
}

template <int N>
__device__ __forceinline__ void regs_inc() {
  asm volatile("setmaxnreg.inc.sync.aligned.u32 %0;" ::"n"(N));
}
template <int N>
__device__ __forceinline__ void regs_dec() {
  asm volatile("setmaxnreg.dec.sync.aligned.u32 %0;" ::"n"(N));
}

// i-th unit of this CTA: rounds of gridDim.x units, alternating direction.
__device__ __forceinline__ int unit_index(int i) {
  const int G = gridDim.x;
  const int c = blockIdx.x;
  return i * G + ((i & 1) ? (G - 1 - c) : c);
}

// Byte offset of the 8-element (16-byte) chunk holding element e (e % 8 == 0)
// of row r in a 128-row tile stored as 128-byte-swizzled column blocks.
__device__ __forceinline__ uint32_t sw128_off(int r, int e) {
  const int blk = e >> 6;
  const int chunk = (e >> 3) & 7;
  return static_cast<uint32_t>(blk * (BM * 128) + r * 128 + ((chunk ^ (r & 7)) << 4));
}

// Rotate row r of a Q tile in shared memory in place (RoPE at position pos).
template <int D>
__device__ __forceinline__ void rotate_q_row(uint8_t* tile, int r, int pos, int layout,
                                             const RopeTable& th) {
#pragma unroll 1
  for (int c = 0; c < D / 16; ++c) {
    int e0, e1;
    if (layout == 1) {
      e0 = 8 * c;
      e1 = D / 2 + 8 * c;
    } else {
      e0 = 16 * c;
      e1 = 16 * c + 8;
    }
    uint4* p0 = reinterpret_cast<uint4*>(tile + sw128_off(r, e0));
    uint4* p1 = reinterpret_cast<uint4*>(tile + sw128_off(r, e1));
    const uint4 a = *p0, b = *p1;
    const uint32_t wa[4] = {a.x, a.y, a.z, a.w};
    const uint32_t wb[4] = {b.x, b.y, b.z, b.w};
    float u[8], w[8];
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      u[2 * i] = bf16lo_to_f32(wa[i]);
      u[2 * i + 1] = bf16hi_to_f32(wa[i]);
      w[2 * i] = bf16lo_to_f32(wb[i]);
      w[2 * i + 1] = bf16hi_to_f32(wb[i]);
    }
    float cs[8], sn[8];
#pragma unroll
    for (int i = 0; i < 8; ++i) rope_cos_sin<false>(pos, th.hi[8 * c + i], th.lo[8 * c + i], cs[i], sn[i]);
    float ou[8], ow[8];
    if (layout == 1) {
#pragma unroll
      for (int i = 0; i < 8; ++i) {
        ou[i] = fmaf(u[i], cs[i], -w[i] * sn[i]);
        ow[i] = fmaf(u[i], sn[i], w[i] * cs[i]);
      }
    } else {
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        ou[2 * i] = fmaf(u[2 * i], cs[i], -u[2 * i + 1] * sn[i]);
        ou[2 * i + 1] = fmaf(u[2 * i], sn[i], u[2 * i + 1] * cs[i]);
        ow[2 * i] = fmaf(w[2 * i], cs[4 + i], -w[2 * i + 1] * sn[4 + i]);
        ow[2 * i + 1] = fmaf(w[2 * i], sn[4 + i], w[2 * i + 1] * cs[4 + i]);
      }
    }
    uint4 ra, rb;
    ra.x = pack_bf16x2(ou[0], ou[1]);
    ra.y = pack_bf16x2(ou[2], ou[3]);
    ra.z = pack_bf16x2(ou[4], ou[5]);
    ra.w = pack_bf16x2(ou[6], ou[7]);
    rb.x = pack_bf16x2(ow[0], ow[1]);
    rb.y = pack_bf16x2(ow[2], ow[3]);
    rb.z = pack_bf16x2(ow[4], ow[5]);
    rb.w = pack_bf16x2(ow[6], ow[7]);
    *p0 = ra;
    *p1 = rb;
  }
}

// S = Q K^T: M=128 query rows, N=128 keys, K=D; both operands K-major,
// 128-byte swizzled; one MMA per 16 channels.
template <int D>
__device__ __forceinline__ void issue_qk(uint32_t d_tmem, uint32_t q_smem, uint32_t k_smem) {
#pragma unroll
  for (int kk = 0; kk < D / 16; ++kk) {
    const uint32_t off = static_cast<uint32_t>((kk >> 2) * (BM * 128) + (kk & 3) * 32);
    umma_ss(d_tmem, smem_desc_sw128(q_smem + off, 16, 1024), smem_desc_sw128(k_smem + off, 16, 1024),
            kIdescS, kk > 0 ? 1u : 0u);
  }
}

// Kernel parameters from the host-side arguments (unit counts, log2-scaled scale).
inline Params make_params(const FwdArgs& a) {
  Params p{};
  p.out = static_cast<__nv_bfloat16*>(a.out);
  p.lse = a.lse;
  p.status = a.status;
  p.B = a.B;
  p.Hq = a.Hq;
  p.Hkv = a.Hkv;
  p.Tq = a.Tq;
  p.Tk = a.Tk;
  p.q_off = a.q_off;
  p.rep = a.Hq / a.Hkv;
  p.hp = p.rep / 2;
  p.n_qt = (a.Tq + BM - 1) / BM;
  p.n_kt = (a.Tk + BN - 1) / BN;
  p.causal = a.causal;
  p.rope = a.rope;
  p.nP = p.n_qt * a.B * a.Hkv * p.hp;
  const int nC = (p.rep & 1) ? ((p.n_qt + 1) / 2) * a.B * a.Hkv : 0;
  p.nUnits = p.nP + nC;
  p.scale_log2 = static_cast<float>(static_cast<double>(a.scale) * 1.4426950408889634);
  p.theta = a.theta;
  p.cache_lens = a.block_table != nullptr ? a.cache_lens : nullptr;
  p.block_table = a.block_table;
  p.page_size = a.page_size;
  p.num_pages = a.num_pages;
  p.max_pages = a.max_pages;
  // rows per K/V box: 128, 64 for an odd multiple of 64, else the page (16 or 32 rows)
  p.box_rows = a.block_table == nullptr || a.page_size % BN == 0
                   ? BN
                   : (a.page_size % 64 == 0 ? 64 : a.page_size);
  return p;
}

}  // namespace fwd
}  // namespace csattn
