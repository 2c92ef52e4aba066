// Gather of a paged KV cache with small pages (16 or 32 rows) into one contiguous
// page per sequence, ahead of the paged prefill: with pages that small a 128-row K
// or V tile would take 4 or 8 TMA boxes and as many block-table reads in the
// prefill kernel's single producer thread, which then sets the pace; one pass that
// copies each sequence's visible rows with 16-byte loads and stores, and the prefill
// kernel over the gathered pages (one box per 64-column block of a tile), is faster.
#include "internal.h"

namespace csattn {
namespace {

constexpr int kGatherThreads = 256;
constexpr int kGatherRows = 32;  // cache rows per CTA

// Rows 0..L_b+Tq-1 (L_b = cache_lens[b]) of KV head g of sequence b go from the page
// pool ([num_pages, Hkv, page_size, d]; row t in page block_table[b * max_pages +
// t / page_size] at offset t % page_size) to rows 0.. of page b of the gathered pools
// ([B, Hkv, Lpad, d]); ident[b] = b is the block table of the gathered pools.  A
// length outside [0, max_pages * page_size - Tq] or a page index outside the pool
// raises kStatusDeviceArg (the rows concerned are zeros or not written).
__global__ void __launch_bounds__(kGatherThreads) gather_pages_kernel(
    const uint4* __restrict__ k_pages, const uint4* __restrict__ v_pages,
    const int32_t* __restrict__ block_table, const int32_t* __restrict__ cache_lens,
    uint4* __restrict__ k_out, uint4* __restrict__ v_out, int32_t* __restrict__ ident, int Hkv,
    int Tq, int d, int page_size, int num_pages, int max_pages, int Lpad, uint32_t* status) {
  const int b = blockIdx.z, g = blockIdx.y, r0 = blockIdx.x * kGatherRows;
  if (g == 0 && blockIdx.x == 0 && threadIdx.x == 0) ident[b] = b;
  int L = cache_lens[b];
  if (L < 0 || L > max_pages * page_size - Tq) {
    if (g == 0 && blockIdx.x == 0 && threadIdx.x == 0) atomicOr(status, kStatusDeviceArg);
    L = 0;
  }
  const int n = L + Tq;
  if (r0 >= n) return;
  const int rows = min(kGatherRows, n - r0);
  const int cpr = d / 8;  // 16-byte chunks per row
  const int per = rows * cpr;
  for (int it = threadIdx.x; it < 2 * per; it += kGatherThreads) {
    const bool is_v = it >= per;
    const int j = is_v ? it - per : it;
    const int r = r0 + j / cpr, c = j - (j / cpr) * cpr;
    const int page = block_table[static_cast<size_t>(b) * max_pages + r / page_size];
    uint4 val = make_uint4(0u, 0u, 0u, 0u);
    if (page >= 0 && page < num_pages) {
      const size_t src =
          ((static_cast<size_t>(page) * Hkv + g) * page_size + r % page_size) * cpr + c;
      val = is_v ? v_pages[src] : k_pages[src];
    } else if (c == 0) {
      atomicOr(status, kStatusDeviceArg);
    }
    const size_t dst = ((static_cast<size_t>(b) * Hkv + g) * Lpad + r) * cpr + c;
    if (is_v)
      v_out[dst] = val;
    else
      k_out[dst] = val;
  }
}

}  // namespace

cudaError_t launch_gather_pages_bf16(const void* k_pages, const void* v_pages,
                                     const int32_t* block_table, const int32_t* cache_lens,
                                     void* k_out, void* v_out, int32_t* ident, int B, int Hkv,
                                     int Tq, int d, int page_size, int num_pages, int max_pages,
                                     int Lpad, uint32_t* status, cudaStream_t stream) {
  dim3 grid((Lpad + kGatherRows - 1) / kGatherRows, Hkv, B);
  gather_pages_kernel<<<grid, kGatherThreads, 0, stream>>>(
      static_cast<const uint4*>(k_pages), static_cast<const uint4*>(v_pages), block_table,
      cache_lens, static_cast<uint4*>(k_out), static_cast<uint4*>(v_out), ident, Hkv, Tq, d,
      page_size, num_pages, max_pages, Lpad, status);
  return cudaGetLastError();
}

}  // namespace csattn
