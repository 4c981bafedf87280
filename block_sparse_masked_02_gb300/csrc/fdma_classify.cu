// Mask-tile classifier (Flash-DMA README, "Key Features": a block is computed
// only when the OR over its mask is true; FlashMask README, "Sparse
// computation": blocks are fully masked, partially masked or unmasked).
//
// For every 128x128 tile it writes
//   - the tile class (0 skip / 1 partial / 2 full) for the attention kernels
//     and, optionally, for the caller;
//   - for tiles the kernels must mask element-wise (partial, or full but cut
//     by the sequence end), two packed keep-bit copies: row-major (forward:
//     one thread per query row reads 16 bytes; bit c%32 of word c/32) and
//     column-major (backward: one thread per key reads 16 bytes; bit r%32 of
//     word r/32).  Bits outside the sequence are zero.
//
// Dense masks (bf16, uint8 or bit-packed): one CTA per tile reads the tile once (bf16: two TMA
// loads into shared memory; uint8 / bit-packed, or a bf16 layout a tensor map cannot describe:
// streaming register loads); each thread owns an 8x8 block, so the column-major copy is one 8x8
// bit transpose per thread.  Column ranges (and no mask): one warp per key tile
// walks a run of query tiles; skip/full follow from per-column masked-row
// counts, and keep bits are built a 32-row word at a time from the ranges.
// Tiles entirely above the causal diagonal are classified without reading.
// Causality is bottom-right aligned: key j is visible from query i when
// j <= i + (Nk - Nq), i.e. the usual j <= i for square problems.
#include "fdma_internal.h"
#include "fdma_ptx.cuh"

namespace fdma {

namespace {

// Keep bits of 8 bf16 mask values (bit e = value e is nonzero; both signed
// zeros count as zero).  (x & 0x7FFF) + 0x7FFF has bit 15 set exactly when the
// magnitude bits are nonzero, with no carry out of the 16-bit half; the two
// halves' top bytes are then gathered and the eight flags packed by one
// multiply whose partial products land on distinct bits.
__device__ __forceinline__ uint32_t keep_byte(const uint4 raw) {
  const uint32_t y0 = (raw.x & 0x7FFF7FFFu) + 0x7FFF7FFFu;
  const uint32_t y1 = (raw.y & 0x7FFF7FFFu) + 0x7FFF7FFFu;
  const uint32_t y2 = (raw.z & 0x7FFF7FFFu) + 0x7FFF7FFFu;
  const uint32_t y3 = (raw.w & 0x7FFF7FFFu) + 0x7FFF7FFFu;
  const uint32_t z01 = __byte_perm(y0, y1, 0x7531);  // flags of values 0..3 at bits 7, 15, 23, 31
  const uint32_t z23 = __byte_perm(y2, y3, 0x7531);  // values 4..7
  const uint32_t w = ((z01 >> 7) & 0x01010101u) | ((z23 >> 3) & 0x10101010u);
  return (w * 0x01020408u) >> 24;
}

// Keep bits of 8 uint8 mask values: bit 7 of (x & 0x7F) + 0x7F, or-ed with x, is set
// exactly when the byte is nonzero; the four top bits of each word are gathered
// the same way as for bf16.
__device__ __forceinline__ uint32_t keep_byte_u8(const uint2 raw) {
  const uint32_t y0 = ((raw.x & 0x7F7F7F7Fu) + 0x7F7F7F7Fu) | raw.x;  // flags of values 0..3 at bits 7, 15, 23, 31
  const uint32_t y1 = ((raw.y & 0x7F7F7F7Fu) + 0x7F7F7F7Fu) | raw.y;  // values 4..7
  const uint32_t w = ((y0 >> 7) & 0x01010101u) | ((y1 >> 3) & 0x10101010u);
  return (w * 0x01020408u) >> 24;
}

// 8x8 bit-matrix transpose (bit 8u+e -> bit 8e+u) by three masked delta swaps
// (Hacker's Delight, section 7-3, "Transposing a Bit Matrix").
__device__ __forceinline__ uint64_t transpose8x8(uint64_t x) {
  uint64_t t = (x ^ (x >> 7)) & 0x00AA00AA00AA00AAull;
  x ^= t ^ (t << 7);
  t = (x ^ (x >> 14)) & 0x0000CCCC0000CCCCull;
  x ^= t ^ (t << 14);
  t = (x ^ (x >> 28)) & 0x00000000F0F0F0F0ull;
  x ^= t ^ (t << 28);
  return x;
}

// 32x32 bit transpose across a warp: lane l holds row l (bit c = column c) and
// gets column l.  Five butterfly stages, each swapping the off-diagonal
// j x j sub-blocks between lanes l and l ^ j (the recursive block transpose of
// Hacker's Delight, section 7-3, spread over lanes).
__device__ __forceinline__ uint32_t transpose32_warp(uint32_t x, int lane) {
#pragma unroll
  for (int j = 16; j >= 1; j >>= 1) {
    const uint32_t m = j == 16 ? 0x0000FFFFu : j == 8 ? 0x00FF00FFu : j == 4 ? 0x0F0F0F0Fu : j == 2 ? 0x33333333u
                                                                                           : 0x55555555u;
    const uint32_t y = __shfl_xor_sync(0xFFFFFFFFu, x, j);
    x = (lane & j) ? ((x & ~m) | ((y >> j) & m)) : ((x & m) | ((y << j) & ~m));
  }
  return x;
}

__device__ __forceinline__ uint32_t low_bits8(int n) { return n >= 8 ? 0xFFu : (n <= 0 ? 0u : (1u << n) - 1u); }
__device__ __forceinline__ uint32_t low_bits32(int n) { return n >= 32 ? 0xFFFFFFFFu : (n <= 0 ? 0u : (1u << n) - 1u); }

__device__ __forceinline__ bool needs_bits(int kcls, bool ragged) {
  return kcls == kPartial || (kcls == kFull && ragged);
}

}  // namespace

// KIND: 0 = bf16 mask, 1 = uint8 / bool mask, 2 = bit-packed mask (one byte per 8 keys).
template <int KIND>
__global__ void __launch_bounds__(256) classify_dense_kernel(const ClassifyParams p) {
  __shared__ __align__(16) uint8_t rowbits[kTile][16];  // bit (c & 7) of byte c >> 3 = keep(q0 + r, k0 + c)
  __shared__ __align__(16) uint8_t colbits[kTile][16];  // bit (r & 7) of byte r >> 3

  const int kt = blockIdx.x, qt = blockIdx.y, bg = blockIdx.z;
  const int b = bg / p.Hkv, g = bg % p.Hkv;
  const int64_t tile = (static_cast<int64_t>(bg) * p.nTq + qt) * p.nTk + kt;
  const int q0 = qt * kTile, k0 = kt * kTile;
  const int tid = threadIdx.x;

  if (p.causal && k0 > q0 + kTile - 1 + p.causal_off && !p.no_skip) {
    if (tid == 0) {
      p.kmap[tile] = kSkip;
      if (p.user_map) p.user_map[tile] = kSkip;
    }
    return;
  }
  const int rows = min(kTile, p.Nq - q0);
  const int cols = min(kTile, p.Nk - k0);
  const bool ragged = rows < kTile || cols < kTile;
  const bool diag = p.causal && k0 + kTile - 1 > q0 + p.causal_off;

  // Thread -> 8x8 block: rows rb*8 .. rb*8+7, columns cc*8 .. cc*8+7.  For each
  // row step a warp reads two whole 256-byte row segments.
  const int cc = tid & 15, rb = tid >> 4;
  const int64_t row_off = b * p.ms_b + g * p.ms_h + static_cast<int64_t>(q0 + rb * 8) * p.ms_r;
  const int64_t off = row_off + k0 + cc * 8;
  const int ncol = cols - cc * 8;  // valid columns of this thread's chunk
  uint64_t blk = 0;                // bit 8u+e = keep(row rb*8+u, column cc*8+e)
  if (KIND == 2) {
    // the mask byte of columns cc*8 .. cc*8+7 is already this block row's keep bits
    const uint8_t* base = p.mask_u8 + row_off + ((k0 + cc * 8) >> 3);
#pragma unroll
    for (int u = 0; u < 8; ++u)
      if (rb * 8 + u < rows && ncol > 0) blk |= static_cast<uint64_t>(base[u * p.ms_r]) << (8 * u);
  } else if (KIND == 1) {
    const uint8_t* base = p.mask_u8 + off;
    uint2 raw[8];
#pragma unroll
    for (int u = 0; u < 8; ++u) {
      raw[u] = make_uint2(0, 0);
      if (rb * 8 + u < rows && ncol > 0) {
        const uint8_t* src = base + u * p.ms_r;
        if (ncol >= 8) {
          raw[u] = __ldcs(reinterpret_cast<const uint2*>(src));
        } else {
          uint32_t h[8] = {0, 0, 0, 0, 0, 0, 0, 0};
          for (int e = 0; e < ncol; ++e) h[e] = src[e];
          raw[u] = make_uint2(h[0] | (h[1] << 8) | (h[2] << 16) | (h[3] << 24),
                              h[4] | (h[5] << 8) | (h[6] << 16) | (h[7] << 24));
        }
      }
    }
#pragma unroll
    for (int u = 0; u < 8; ++u) blk |= static_cast<uint64_t>(keep_byte_u8(raw[u])) << (8 * u);
  } else {
    const uint16_t* base = p.mask + off;
    uint4 raw[8];
#pragma unroll
    for (int u = 0; u < 8; ++u) {
      raw[u] = make_uint4(0, 0, 0, 0);
      if (rb * 8 + u < rows && ncol > 0) {
        const uint16_t* src = base + u * p.ms_r;
        if (ncol >= 8) {
          raw[u] = __ldcs(reinterpret_cast<const uint4*>(src));
        } else {
          uint32_t h[8] = {0, 0, 0, 0, 0, 0, 0, 0};
          for (int e = 0; e < ncol; ++e) h[e] = src[e];
          raw[u] = make_uint4(h[0] | (h[1] << 16), h[2] | (h[3] << 16), h[4] | (h[5] << 16), h[6] | (h[7] << 16));
        }
      }
    }
#pragma unroll
    for (int u = 0; u < 8; ++u) blk |= static_cast<uint64_t>(keep_byte(raw[u])) << (8 * u);
  }

  uint64_t valid = ~0ull;
  if (ragged || diag) {
    const uint32_t cmask = low_bits8(ncol);
    valid = 0;
#pragma unroll
    for (int u = 0; u < 8; ++u) {
      const int r = rb * 8 + u;
      const uint32_t vm = r < rows ? cmask : 0u;
      valid |= static_cast<uint64_t>(vm) << (8 * u);
      // causal: keep only columns j <= i + off, i.e. c <= r + q0 + off - k0
      const uint32_t cm = diag ? low_bits8(r + q0 + p.causal_off - k0 - cc * 8 + 1) : 0xFFu;
      blk &= ~(static_cast<uint64_t>(0xFFu & ~(vm & cm)) << (8 * u));
    }
  }

  // Stage both bit copies; the rotations keep the byte stores of a warp on
  // distinct banks.
  const uint64_t tr = transpose8x8(blk);
#pragma unroll
  for (int s = 0; s < 8; ++s) {
    const int u = (s + 4 * (rb & 1)) & 7;
    rowbits[rb * 8 + u][cc] = static_cast<uint8_t>(blk >> (8 * u));
    const int e = (s + cc) & 7;
    colbits[cc * 8 + e][rb] = static_cast<uint8_t>(tr >> (8 * e));
  }
  const int any = __syncthreads_or(blk != 0);
  const int all = __syncthreads_and((blk | ~valid) == ~0ull);
  const int cls = any ? (all ? kFull : kPartial) : kSkip;
  const int kcls = p.no_skip ? kPartial : cls;
  if (tid == 0) {
    p.kmap[tile] = static_cast<int8_t>(kcls);
    if (p.user_map) p.user_map[tile] = static_cast<int8_t>(cls);
  }
  if (!needs_bits(kcls, ragged)) return;
  if (tid < kTile)
    p.bits_row[tile * kTile + tid] = *reinterpret_cast<const uint4*>(rowbits[tid]);
  else
    p.bits_col[tile * kTile + tid - kTile] = *reinterpret_cast<const uint4*>(colbits[tid - kTile]);
}

// bf16 masks: the same per-tile work, but the 32 KB mask tile arrives by two TMA loads (64-key
// SW128 boxes; out-of-range rows and keys read as zeros) into shared memory, and each thread
// reads its 8x8 block from there.  32 registers and 36 KB of shared memory per CTA: six tiles'
// loads in flight per SM (6 % faster than the register loads at N=16384).
constexpr uint32_t kClsTmaSmem = 32768 + 2048 + 2048 + 16;  // tile, row bits, column bits, barrier
__global__ void __launch_bounds__(256)
    classify_tma1_kernel(const __grid_constant__ CUtensorMap tmM, const ClassifyParams p) {
  extern __shared__ __align__(1024) uint8_t smem[];
  uint8_t(*rowbits)[16] = reinterpret_cast<uint8_t(*)[16]>(smem + 32768);
  uint8_t(*colbits)[16] = reinterpret_cast<uint8_t(*)[16]>(smem + 34816);
  uint64_t& full = *reinterpret_cast<uint64_t*>(smem + 36864);
  const int kt = blockIdx.x, qt = blockIdx.y, bg = blockIdx.z;
  const int b = bg / p.Hkv, g = bg % p.Hkv;
  const int64_t tile = (static_cast<int64_t>(bg) * p.nTq + qt) * p.nTk + kt;
  const int q0 = qt * kTile, k0 = kt * kTile;
  const int tid = threadIdx.x;
  if (p.causal && k0 > q0 + kTile - 1 + p.causal_off && !p.no_skip) {
    if (tid == 0) {
      p.kmap[tile] = kSkip;
      if (p.user_map) p.user_map[tile] = kSkip;
    }
    return;
  }
  if ((smem_u32(smem) & 1023u) != 0) {
    if (tid == 0) atomicCAS(p.err, 0, kDevErrAlign);
    return;
  }
  if (tid == 0) {
    mbar_init(&full, 1);
    fence_mbar_init();
    mbar_arrive_expect_tx(&full, 32768);
    tma_load_4d(smem, &tmM, &full, k0, q0, g * p.mask_hsel, b * p.mask_bsel);
    tma_load_4d(smem + 16384, &tmM, &full, k0 + 64, q0, g * p.mask_hsel, b * p.mask_bsel);
  }
  __syncthreads();
  const bool got = mbar_wait(&full, 0, p.err, kDevErrTimeout, nullptr);  // bounded; on time-out the error is set
  const int rows = min(kTile, p.Nq - q0);
  const int cols = min(kTile, p.Nk - k0);
  const bool ragged = rows < kTile || cols < kTile;
  const bool diag = p.causal && k0 + kTile - 1 > q0 + p.causal_off;
  const int cc = tid & 15, rb = tid >> 4;
  const int ncol = cols - cc * 8;
  const uint8_t* tb = smem + (cc >> 3) * 16384;  // row r's 16-byte chunk j sits at chunk j ^ (r & 7)
  uint64_t blk = 0;
  if (got) {
#pragma unroll
    for (int u = 0; u < 8; ++u) {
      const int r = rb * 8 + u;
      const uint4 raw = *reinterpret_cast<const uint4*>(tb + r * 128 + (((cc & 7) ^ (r & 7)) << 4));
      blk |= static_cast<uint64_t>(keep_byte(raw)) << (8 * u);
    }
  }
  uint64_t valid = ~0ull;
  if (ragged || diag) {
    const uint32_t cmask = low_bits8(ncol);
    valid = 0;
#pragma unroll
    for (int u = 0; u < 8; ++u) {
      const int r = rb * 8 + u;
      const uint32_t vm = r < rows ? cmask : 0u;
      valid |= static_cast<uint64_t>(vm) << (8 * u);
      const uint32_t cm = diag ? low_bits8(r + q0 + p.causal_off - k0 - cc * 8 + 1) : 0xFFu;
      blk &= ~(static_cast<uint64_t>(0xFFu & ~(vm & cm)) << (8 * u));
    }
  }
  const uint64_t tr = transpose8x8(blk);
#pragma unroll
  for (int s = 0; s < 8; ++s) {
    const int u = (s + 4 * (rb & 1)) & 7;
    rowbits[rb * 8 + u][cc] = static_cast<uint8_t>(blk >> (8 * u));
    const int e = (s + cc) & 7;
    colbits[cc * 8 + e][rb] = static_cast<uint8_t>(tr >> (8 * e));
  }
  const int any = __syncthreads_or(blk != 0);
  const int all = __syncthreads_and((blk | ~valid) == ~0ull);
  const int cls = any ? (all ? kFull : kPartial) : kSkip;
  const int kcls = p.no_skip ? kPartial : cls;
  if (tid == 0) {
    p.kmap[tile] = static_cast<int8_t>(kcls);
    if (p.user_map) p.user_map[tile] = static_cast<int8_t>(cls);
  }
  if (!needs_bits(kcls, ragged)) return;
  if (tid < kTile)
    p.bits_row[tile * kTile + tid] = *reinterpret_cast<const uint4*>(rowbits[tid]);
  else
    p.bits_col[tile * kTile + tid - kTile] = *reinterpret_cast<const uint4*>(colbits[tid - kTile]);
}

cudaError_t launch_classify_tma1(const CUtensorMap& tm, const ClassifyParams& p, cudaStream_t stream) {
  cudaError_t e = cudaFuncSetAttribute(classify_tma1_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, kClsTmaSmem);
  if (e != cudaSuccess) return e;
  const dim3 grid(p.nTk, p.nTq, p.B * p.Hkv);
  classify_tma1_kernel<<<grid, 256, kClsTmaSmem, stream>>>(tm, p);
  return cudaGetLastError();
}

// One warp per (batch, kv head, key tile) and run of kRangeChunk query tiles;
// lane l owns columns l + 32*s.
constexpr int kRangeChunk = 16;

__global__ void __launch_bounds__(256) classify_ranges_kernel(const ClassifyParams p) {
  const int lane = threadIdx.x & 31;
  const int nchunk = (p.nTq + kRangeChunk - 1) / kRangeChunk;
  const int64_t wid = static_cast<int64_t>(blockIdx.x) * 8 + (threadIdx.x >> 5);
  if (wid >= static_cast<int64_t>(p.B) * p.Hkv * p.nTk * nchunk) return;
  const int64_t strip = wid / nchunk;
  const int qt_begin = static_cast<int>(wid % nchunk) * kRangeChunk;
  const int qt_end = min(p.nTq, qt_begin + kRangeChunk);
  const int kt = static_cast<int>(strip % p.nTk);
  const int bg = static_cast<int>(strip / p.nTk);
  const int b = bg / p.Hkv, g = bg % p.Hkv;
  const int k0 = kt * kTile, cols = min(kTile, p.Nk - k0);

  // Masked rows of column c are [lo, hi) and (second kind) [lo2, hi2), clamped to
  // [0, Nq] (a range is empty when hi <= lo).
  const bool two = p.mask_kind == FDMA_MASK_COLRANGES2;
  const int per = two ? 4 : 2;
  int lo[4], hi[4], lo2[4], hi2[4];
#pragma unroll
  for (int s = 0; s < 4; ++s) {
    lo[s] = hi[s] = lo2[s] = hi2[s] = 0;
    const int c = lane + 32 * s;
    if (p.mask_kind != FDMA_MASK_NONE && c < cols) {
      const int32_t* src = p.cr + b * p.cr_b + g * p.cr_h + per * static_cast<int64_t>(k0 + c);
      lo[s] = min(max(src[0], 0), p.Nq);
      hi[s] = min(max(src[1], 0), p.Nq);
      if (two) {
        lo2[s] = min(max(src[2], 0), p.Nq);
        hi2[s] = min(max(src[3], 0), p.Nq);
      }
    }
  }

  for (int qt = qt_begin; qt < qt_end; ++qt) {
    const int q0 = qt * kTile, rows = min(kTile, p.Nq - q0);
    const int64_t tile = (static_cast<int64_t>(bg) * p.nTq + qt) * p.nTk + kt;
    const bool ragged = rows < kTile || cols < kTile;
    const bool above = p.causal && k0 > q0 + kTile - 1 + p.causal_off;
    const bool diag = p.causal && k0 + kTile - 1 > q0 + p.causal_off;  // includes "above"
    int cls = kSkip;
    bool exact = false;  // class known without keep bits
    if (above && !p.no_skip) {
      exact = true;
    } else if (!diag && !p.no_skip) {
      bool kept = true, masked = true;
#pragma unroll
      for (int s = 0; s < 4; ++s) {
        if (lane + 32 * s < cols) {
          // masked rows of the tile: |R1 ∩ T| + |R2 ∩ T| - |R1 ∩ R2 ∩ T|
          const int q1 = q0 + rows;
          int m = max(0, min(hi[s], q1) - max(lo[s], q0));
          if (two) {
            m += max(0, min(hi2[s], q1) - max(lo2[s], q0));
            m -= max(0, min(min(hi[s], hi2[s]), q1) - max(max(lo[s], lo2[s]), q0));
          }
          kept &= m == 0;
          masked &= m == rows;
        }
      }
      kept = __all_sync(0xFFFFFFFFu, kept);
      masked = __all_sync(0xFFFFFFFFu, masked);
      cls = masked ? kSkip : (kept ? kFull : kPartial);
      exact = !needs_bits(cls, ragged);
    }
    if (!exact) {
      uint32_t cb[4][4];  // [column slot][row word]: bit r of word w = keep(q0 + 32w + r, column)
      bool any = false, all = true;
#pragma unroll
      for (int s = 0; s < 4; ++s) {
        const int c = lane + 32 * s;
#pragma unroll
        for (int w = 0; w < 4; ++w) {
          const int r0 = q0 + 32 * w;
          uint32_t vm = 0, word = 0;
          if (c < cols) {
            vm = low_bits32(rows - 32 * w);
            word = vm & ~(low_bits32(hi[s] - r0) & ~low_bits32(lo[s] - r0));
            if (two) word &= ~(low_bits32(hi2[s] - r0) & ~low_bits32(lo2[s] - r0));
            if (p.causal) word &= ~low_bits32(k0 + c - p.causal_off - r0);  // keep rows i >= j - off
          }
          any |= word != 0;
          all &= word == vm;
          cb[s][w] = word;
        }
      }
      any = __any_sync(0xFFFFFFFFu, any);
      all = __all_sync(0xFFFFFFFFu, all);
      cls = any ? (all ? kFull : kPartial) : kSkip;
      const int kcls = p.no_skip ? kPartial : cls;
      if (needs_bits(kcls, ragged)) {
#pragma unroll
        for (int s = 0; s < 4; ++s)
          p.bits_col[tile * kTile + lane + 32 * s] = make_uint4(cb[s][0], cb[s][1], cb[s][2], cb[s][3]);
        // row-major copy: word s of row 32w + lane = bit lane of every lane's cb[s][w]
#pragma unroll
        for (int w = 0; w < 4; ++w) {
          uint32_t o[4];
#pragma unroll
          for (int s = 0; s < 4; ++s) o[s] = transpose32_warp(cb[s][w], lane);
          p.bits_row[tile * kTile + 32 * w + lane] = make_uint4(o[0], o[1], o[2], o[3]);
        }
      }
    }
    if (lane == 0) {
      p.kmap[tile] = static_cast<int8_t>(p.no_skip ? kPartial : cls);
      if (p.user_map) p.user_map[tile] = static_cast<int8_t>(cls);
    }
  }
}

cudaError_t launch_classify(const ClassifyParams& p, cudaStream_t stream) {
  if (p.mask_kind == FDMA_MASK_DENSE || p.mask_kind == FDMA_MASK_DENSE_U8 || p.mask_kind == FDMA_MASK_BITS) {
    dim3 grid(p.nTk, p.nTq, p.B * p.Hkv);
    if (p.mask_kind == FDMA_MASK_DENSE_U8)
      classify_dense_kernel<1><<<grid, 256, 0, stream>>>(p);
    else if (p.mask_kind == FDMA_MASK_BITS)
      classify_dense_kernel<2><<<grid, 256, 0, stream>>>(p);
    else
      classify_dense_kernel<0><<<grid, 256, 0, stream>>>(p);
  } else {
    const int64_t warps = static_cast<int64_t>(p.B) * p.Hkv * p.nTk * ((p.nTq + kRangeChunk - 1) / kRangeChunk);
    classify_ranges_kernel<<<static_cast<unsigned>((warps + 7) / 8), 256, 0, stream>>>(p);
  }
  return cudaGetLastError();
}

}  // namespace fdma
