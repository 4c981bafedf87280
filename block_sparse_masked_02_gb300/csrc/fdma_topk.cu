// Dynamic top-k mask generation (Flash-DMA README, "Quick Start" example: per query
// row keep the keep_window keys of largest bias, drop the kept keys whose bias is the
// dtype minimum, scatter 1 there, then masked_fill the bias with the dtype minimum
// wherever the mask is 0).
//
// One CTA per row.  The row's bf16 values are turned into 16-bit keys whose unsigned
// order is the numeric order (+0 and -0 map to the same key) and kept in shared memory.
// The k-th largest key t is found by a two-digit radix select (the top 12 bits over a
// 4096-bin histogram, then the low 4 bits of the keys in the chosen bin); keys above t
// are kept, and of the keys equal to t the ones with the smallest key indices, ranked by
// a block-wide scan in index order.
#include "fdma_internal.h"

namespace fdma {
namespace {

constexpr int kTopkThreads = 512;
constexpr int kTopkWarps = kTopkThreads / 32;
constexpr int kTopkVec = 8;  // bf16 values per thread and round (16 bytes)
constexpr uint16_t kBf16Min = 0xFF7Fu;
constexpr uint16_t kBf16One = 0x3F80u;

// Unsigned key with the numeric order of the bf16 value (NaN-free input).
__device__ __forceinline__ uint32_t order_key(uint32_t x) {
  x = (x == 0x8000u) ? 0u : x;  // -0 == +0
  return (x & 0x8000u) ? (~x & 0xFFFFu) : (x | 0x8000u);
}

// Exclusive prefix sum of v over the CTA (index order = thread order); also returns the total.
__device__ __forceinline__ uint32_t block_exclusive_scan(uint32_t v, uint32_t* sWarp, uint32_t& total) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  uint32_t x = v;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const uint32_t y = __shfl_up_sync(0xffffffffu, x, o);
    if (lane >= o) x += y;
  }
  if (lane == 31) sWarp[warp] = x;
  __syncthreads();
  if (warp == 0) {
    uint32_t w = lane < kTopkWarps ? sWarp[lane] : 0u;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const uint32_t y = __shfl_up_sync(0xffffffffu, w, o);
      if (lane >= o) w += y;
    }
    if (lane < kTopkWarps) sWarp[lane] = w;  // inclusive prefix over warps
  }
  __syncthreads();
  const uint32_t before = (warp > 0 ? sWarp[warp - 1] : 0u) + x - v;
  total = sWarp[kTopkWarps - 1];
  __syncthreads();  // sWarp is reused by the next scan
  return before;
}

// Finds the bin of sHist[0..nbins) (nbins = 8 * threads or fewer, counted from the top
// bin down) that holds the need-th largest element, and the count of elements in the
// bins above it; results in sSel[0], sSel[1].
__device__ __forceinline__ void select_bin(const uint32_t* sHist, int nbins, uint32_t need, uint32_t* sWarp,
                                           uint32_t* sSel) {
  // thread t owns bins top-8t .. top-8t-7 (descending)
  const int top = nbins - 1 - 8 * static_cast<int>(threadIdx.x);
  uint32_t c[8], tot = 0;
#pragma unroll
  for (int e = 0; e < 8; ++e) {
    c[e] = (top - e >= 0) ? sHist[top - e] : 0u;
    tot += c[e];
  }
  uint32_t all;
  uint32_t above = block_exclusive_scan(tot, sWarp, all);
  if (above < need && need <= above + tot) {
#pragma unroll
    for (int e = 0; e < 8; ++e) {
      if (above < need && need <= above + c[e]) {
        sSel[0] = static_cast<uint32_t>(top - e);
        sSel[1] = above;
      }
      above += c[e];
    }
  }
  __syncthreads();
}

__global__ void __launch_bounds__(kTopkThreads) topk_mask_kernel(const TopkParams p) {
  extern __shared__ __align__(16) uint8_t smem[];
  uint32_t* sHist = reinterpret_cast<uint32_t*>(smem);          // [4096]
  uint32_t* sWarp = sHist + 4096;                                // [32]
  uint32_t* sSel = sWarp + 32;                                   // [4]
  uint16_t* sKey = reinterpret_cast<uint16_t*>(sSel + 4);        // [Nk]

  const int tid = threadIdx.x;
  const int64_t row = blockIdx.x;
  const int i = static_cast<int>(row % p.Nq);
  const int64_t bg = row / p.Nq;
  const int g = static_cast<int>(bg % p.Hkv);
  const int b = static_cast<int>(bg / p.Hkv);
  const int64_t src_off = b * p.bias_stride[0] + g * p.bias_stride[1] + i * p.bias_stride[2];
  const uint16_t* src = p.bias + src_off;
  uint16_t* bout = p.bias_out != nullptr ? p.bias_out + src_off : nullptr;
  const int64_t dst_off = row * p.Nk;
  const int nround = p.Nk / (kTopkThreads * kTopkVec) + ((p.Nk % (kTopkThreads * kTopkVec)) != 0);

  if (p.keep >= p.Nk) {  // every key kept (the example builds no top-k then)
    for (int r = 0; r < nround; ++r) {
      const int j0 = (r * kTopkThreads + tid) * kTopkVec;
      if (j0 >= p.Nk) break;
      const uint4 v = *reinterpret_cast<const uint4*>(src + j0);
      if (p.mask_u8) *reinterpret_cast<uint2*>(p.mask_u8 + dst_off + j0) = make_uint2(0x01010101u, 0x01010101u);
      else {
        const uint32_t one2 = (static_cast<uint32_t>(kBf16One) << 16) | kBf16One;
        *reinterpret_cast<uint4*>(p.mask_bf16 + dst_off + j0) = make_uint4(one2, one2, one2, one2);
      }
      if (bout != nullptr && bout != src) *reinterpret_cast<uint4*>(bout + j0) = v;
    }
    return;
  }

  // ---- keys into shared memory; histogram of their top 12 bits
  for (int e = tid; e < 4096; e += kTopkThreads) sHist[e] = 0u;
  __syncthreads();
  for (int r0 = 0; r0 < nround; r0 += 4) {
    uint4 v[4];
#pragma unroll
    for (int u = 0; u < 4; ++u) {  // four rounds of loads in flight
      const int j0 = ((r0 + u) * kTopkThreads + tid) * kTopkVec;
      if (r0 + u < nround && j0 < p.Nk) v[u] = *reinterpret_cast<const uint4*>(src + j0);
    }
#pragma unroll
    for (int u = 0; u < 4; ++u) {
      const int j0 = ((r0 + u) * kTopkThreads + tid) * kTopkVec;
      if (r0 + u >= nround || j0 >= p.Nk) break;
      const uint32_t w[4] = {v[u].x, v[u].y, v[u].z, v[u].w};
      uint32_t k2[4];
#pragma unroll
      for (int q = 0; q < 4; ++q) {
        const uint32_t lo = order_key(w[q] & 0xFFFFu), hi = order_key(w[q] >> 16);
        k2[q] = lo | (hi << 16);
        atomicAdd(&sHist[lo >> 4], 1u);
        atomicAdd(&sHist[hi >> 4], 1u);
      }
      *reinterpret_cast<uint4*>(sKey + j0) = make_uint4(k2[0], k2[1], k2[2], k2[3]);
    }
  }
  __syncthreads();
  select_bin(sHist, 4096, static_cast<uint32_t>(p.keep), sWarp, sSel);
  const uint32_t hb = sSel[0], above_hb = sSel[1];

  // ---- histogram of the low 4 bits of the keys in bin hb
  if (tid < 16) sHist[tid] = 0u;
  __syncthreads();
  for (int j = tid * 2; j < p.Nk; j += kTopkThreads * 2) {
    const uint32_t kk = *reinterpret_cast<const uint32_t*>(sKey + j);
    if (((kk & 0xFFFFu) >> 4) == hb) atomicAdd(&sHist[kk & 0xFu], 1u);
    if ((kk >> 20) == hb) atomicAdd(&sHist[(kk >> 16) & 0xFu], 1u);
  }
  __syncthreads();
  select_bin(sHist, 16, static_cast<uint32_t>(p.keep) - above_hb, sWarp, sSel);
  const uint32_t t = (hb << 4) | sSel[0];
  const uint32_t need_eq = static_cast<uint32_t>(p.keep) - above_hb - sSel[1];  // keys equal to t to keep (>= 1)

  // ---- outputs, in index order; ties at t ranked by a scan per round
  uint32_t eq_before = 0;  // keys equal to t in earlier rounds
  for (int r = 0; r < nround; ++r) {
    const int j0 = (r * kTopkThreads + tid) * kTopkVec;
    const bool in = j0 < p.Nk;
    uint16_t kk[kTopkVec];
    uint32_t n_eq = 0;
    if (in) {
      const uint4 kv = *reinterpret_cast<const uint4*>(sKey + j0);
      const uint32_t w[4] = {kv.x, kv.y, kv.z, kv.w};
#pragma unroll
      for (int q = 0; q < 4; ++q) {
        kk[2 * q] = static_cast<uint16_t>(w[q] & 0xFFFFu);
        kk[2 * q + 1] = static_cast<uint16_t>(w[q] >> 16);
      }
#pragma unroll
      for (int e = 0; e < kTopkVec; ++e) n_eq += kk[e] == t;
    }
    uint32_t round_eq;
    uint32_t rank = eq_before + block_exclusive_scan(n_eq, sWarp, round_eq);
    eq_before += round_eq;
    if (!in) continue;
    const uint4 v = *reinterpret_cast<const uint4*>(src + j0);
    const uint32_t w[4] = {v.x, v.y, v.z, v.w};
    uint32_t bo[4], mo[4], m8[2] = {0u, 0u};
#pragma unroll
    for (int q = 0; q < 4; ++q) {
      uint32_t outw = 0, maskw = 0;
#pragma unroll
      for (int h = 0; h < 2; ++h) {
        const int e = 2 * q + h;
        const uint32_t val = (w[q] >> (16 * h)) & 0xFFFFu;
        bool kept = kk[e] > t;
        if (kk[e] == t) kept = rank++ < need_eq;
        kept = kept && val != kBf16Min;
        outw |= (kept ? val : kBf16Min) << (16 * h);
        maskw |= (kept ? kBf16One : 0u) << (16 * h);
        m8[e >> 2] |= (kept ? 1u : 0u) << (8 * (e & 3));
      }
      bo[q] = outw;
      mo[q] = maskw;
    }
    if (p.mask_u8) *reinterpret_cast<uint2*>(p.mask_u8 + dst_off + j0) = make_uint2(m8[0], m8[1]);
    else *reinterpret_cast<uint4*>(p.mask_bf16 + dst_off + j0) = make_uint4(mo[0], mo[1], mo[2], mo[3]);
    if (bout != nullptr) *reinterpret_cast<uint4*>(bout + j0) = make_uint4(bo[0], bo[1], bo[2], bo[3]);
  }
}

}  // namespace

size_t topk_smem_bytes(int Nk) { return (4096 + 32 + 4) * 4 + static_cast<size_t>(Nk) * 2; }

cudaError_t launch_topk(const TopkParams& p, cudaStream_t stream) {
  const size_t smem = topk_smem_bytes(p.Nk);
  cudaError_t e = cudaFuncSetAttribute(topk_mask_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       static_cast<int>(smem));
  if (e != cudaSuccess) return e;
  const int64_t rows = static_cast<int64_t>(p.B) * p.Hkv * p.Nq;
  if (rows == 0) return cudaSuccess;
  topk_mask_kernel<<<static_cast<unsigned>(rows), kTopkThreads, smem, stream>>>(p);
  return cudaGetLastError();
}

}  // namespace fdma
