// Mask-tile classifier (Flash-DMA README, "Key Features": a block is computed
// only when the OR over its mask is true; FlashMask README, "Sparse
// computation": blocks are fully masked, partially masked or unmasked).
//
// One CTA per 128x128 tile.  It reads the tile's dense mask once (16-byte
// streaming loads), or evaluates the column ranges, ANDs in causality and the
// bounds, and writes
//   - the tile class (0 skip / 1 partial / 2 full) for the attention kernels
//     and, optionally, for the caller;
//   - for tiles the kernels must mask element-wise (partial, or cut by the
//     sequence end), two packed keep-bit copies: row-major (forward: one
//     thread per query row reads 16 bytes) and column-major (backward: one
//     thread per key reads 16 bytes).
// Tiles entirely above the causal diagonal are classified without reading.
#include "fdma_internal.h"

namespace fdma {

__global__ void __launch_bounds__(256) classify_kernel(const ClassifyParams p) {
  __shared__ uint8_t rowbits[kTile][16];  // bit (c & 7) of byte c >> 3 = keep(q0 + r, k0 + c)
  __shared__ int2 ranges[kTile];

  const int kt = blockIdx.x, qt = blockIdx.y, bg = blockIdx.z;
  const int b = bg / p.Hkv, g = bg % p.Hkv;
  const int64_t tile = (static_cast<int64_t>(bg) * p.nTq + qt) * p.nTk + kt;
  const int q0 = qt * kTile, k0 = kt * kTile;
  const int tid = threadIdx.x;

  if (p.causal && k0 > q0 + kTile - 1 && !p.no_skip) {
    if (tid == 0) {
      p.kmap[tile] = kSkip;
      if (p.user_map) p.user_map[tile] = kSkip;
    }
    return;
  }
  const int rows = min(kTile, p.Nq - q0);
  const int cols = min(kTile, p.Nk - k0);
  const bool ragged = rows < kTile || cols < kTile;

  // Column ranges / no mask away from the causal diagonal: each column masks one
  // contiguous run of the tile's rows, so the class follows from 128 per-column
  // counts; only partial (or ragged) tiles need the per-element pass below.
  if (p.mask_kind != FDMA_MASK_DENSE && !p.no_skip && !(p.causal && k0 + kTile - 1 > q0)) {
    int masked = 0;
    if (p.mask_kind == FDMA_MASK_COLRANGES && tid < cols) {
      const int32_t* src = p.cr + b * p.cr_b + g * p.cr_h + 2 * static_cast<int64_t>(k0 + tid);
      const int lo = max(src[0], q0), hi = min(src[1], q0 + rows);
      masked = max(0, hi - lo);
    }
    const int all_kept = __syncthreads_and(tid >= cols || masked == 0);
    const int all_masked = __syncthreads_and(tid >= cols || masked == rows);
    const int cls = all_masked ? kSkip : (all_kept ? kFull : kPartial);
    if (cls == kSkip || (cls == kFull && !ragged)) {
      if (tid == 0) {
        p.kmap[tile] = static_cast<int8_t>(cls);
        if (p.user_map) p.user_map[tile] = static_cast<int8_t>(cls);
      }
      return;
    }
  }

  if (p.mask_kind == FDMA_MASK_COLRANGES) {
    if (tid < kTile) {
      int2 rg = make_int2(0, 0);
      if (tid < cols) {
        const int32_t* src = p.cr + b * p.cr_b + g * p.cr_h + 2 * static_cast<int64_t>(k0 + tid);
        rg = make_int2(src[0], src[1]);
      }
      ranges[tid] = rg;
    }
    __syncthreads();
  }

  // 2048 chunks of 8 columns; thread tid owns chunks tid + 256*u.
  int any = 0, all = 1;
  uint4 raw[8];
#pragma unroll
  for (int u = 0; u < 8; ++u) raw[u] = make_uint4(0, 0, 0, 0);
  if (p.mask_kind == FDMA_MASK_DENSE) {
#pragma unroll
    for (int u = 0; u < 8; ++u) {
      const int idx = tid + 256 * u, r = idx >> 4, cc = idx & 15;
      if (r < rows && cc * 8 < cols) {
        const uint16_t* src = p.mask + b * p.ms_b + g * p.ms_h + static_cast<int64_t>(q0 + r) * p.ms_r + k0 + cc * 8;
        if (cc * 8 + 8 <= cols) {
          raw[u] = __ldcs(reinterpret_cast<const uint4*>(src));
        } else {
          uint16_t tmp[8] = {0, 0, 0, 0, 0, 0, 0, 0};
          for (int e = 0; e < cols - cc * 8; ++e) tmp[e] = src[e];
          raw[u] = make_uint4(tmp[0] | (uint32_t(tmp[1]) << 16), tmp[2] | (uint32_t(tmp[3]) << 16),
                              tmp[4] | (uint32_t(tmp[5]) << 16), tmp[6] | (uint32_t(tmp[7]) << 16));
        }
      }
    }
  }
#pragma unroll
  for (int u = 0; u < 8; ++u) {
    const int idx = tid + 256 * u, r = idx >> 4, cc = idx & 15;
    const int i = q0 + r;
    uint32_t byte = 0;
    if (r < rows) {
      const uint32_t w[4] = {raw[u].x, raw[u].y, raw[u].z, raw[u].w};
#pragma unroll
      for (int e = 0; e < 8; ++e) {
        const int c = cc * 8 + e, j = k0 + c;
        if (c < cols) {
          bool keep;
          if (p.mask_kind == FDMA_MASK_DENSE) {
            const uint32_t h = (w[e >> 1] >> ((e & 1) * 16)) & 0xFFFFu;
            keep = (h & 0x7FFFu) != 0;  // nonzero (either sign of zero counts as zero)
          } else if (p.mask_kind == FDMA_MASK_COLRANGES) {
            const int2 rg = ranges[c];
            keep = !(rg.x <= i && i < rg.y);
          } else {
            keep = true;
          }
          if (p.causal) keep = keep && (j <= i);
          byte |= static_cast<uint32_t>(keep) << e;
          any |= keep;
          all &= keep;
        }
      }
    }
    rowbits[r][cc] = static_cast<uint8_t>(byte);
  }
  any = __syncthreads_or(any);
  all = __syncthreads_and(all);
  const int cls = any ? (all ? kFull : kPartial) : kSkip;
  const int kcls = p.no_skip ? kPartial : cls;
  if (tid == 0) {
    p.kmap[tile] = static_cast<int8_t>(kcls);
    if (p.user_map) p.user_map[tile] = static_cast<int8_t>(cls);
  }
  if (kcls == kSkip || (kcls == kFull && !ragged)) return;

  if (tid < kTile) p.bits_row[tile * kTile + tid] = *reinterpret_cast<const uint4*>(rowbits[tid]);
  // column-major: thread -> (column c, half h of the rows)
  const int c = tid >> 1, h = tid & 1;
  uint32_t lo = 0, hi = 0;
#pragma unroll 8
  for (int rr = 0; rr < 32; ++rr) {
    lo |= static_cast<uint32_t>((rowbits[h * 64 + rr][c >> 3] >> (c & 7)) & 1u) << rr;
    hi |= static_cast<uint32_t>((rowbits[h * 64 + 32 + rr][c >> 3] >> (c & 7)) & 1u) << rr;
  }
  reinterpret_cast<uint2*>(&p.bits_col[tile * kTile + c])[h] = make_uint2(lo, hi);
}

cudaError_t launch_classify(const ClassifyParams& p, cudaStream_t stream) {
  dim3 grid(p.nTk, p.nTq, p.B * p.Hkv);
  classify_kernel<<<grid, 256, 0, stream>>>(p);
  return cudaGetLastError();
}

}  // namespace fdma
