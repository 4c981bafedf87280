// Backward for the wide head dims (d, dv) = (192, 128) and (256, 256) (FlashMask README,
// "Performance": the SM100 head-dim table lists both).  The gradients are the same as for the
// narrower heads (Flash-DMA issue #73, "Project Progress": the backward reuses the forward's
// mask / bias handling and adds dBias); only the plan differs.
//
// At d = 128 one CTA keeps S^T, dP^T, dV and dK (4 x 128 columns) in TMEM; wider heads do not
// fit.  Here the output columns are split into parts of at most 128: part P (one launch each)
// owns dK / dQ columns [128P, 128P + KW) and dV columns [128P, 128P + VW) (192 / 128: part 0
// 128 / 128, part 1 64 / 0; 256 / 256: 128 / 128 twice).  Every CTA of a part recomputes
// S^T = K Q^T and dP^T = V dO^T over the full widths and accumulates only its own columns:
//   TMEM   S^T / P^T 0..127, dP^T and then dQ 128..255, dV 256.., dK 384..
//   smem   Q (full width); at 192 / 128 all of K and V resident and X holding dO; at 256 / 256
//          the part's K columns resident, a buffer X that holds the other K columns until S^T
//          has read them and then dO, and a two-slot ring that streams V in 64-column chunks;
//          and a buffer that holds a query tile's bias until the compute warps have copied it
//          into registers and then each step's dS^T.
// One CTA = (batch, kv head, 128-key tile) of one part.  Roles: warp 0 TMA producer, warp 1
// MMA issuer, warps 4..11 two compute warpgroups (keys on TMEM lanes, 64 queries each; P pass,
// then dS pass), warps 12..15 dQ drain (fp32 reductions into the (B, nqpad, Hq, d) accumulator).
// Each step runs S^T, dP^T, dV, dQ, dK in that order with little overlap: this path is for
// coverage of the wide head dims, the d <= 128 kernel is the fast one.
#include "fdma_internal.h"
#include "fdma_ptx.cuh"

namespace fdma {
namespace {

constexpr float kLog2eW = 1.4426950408889634f;

__device__ __forceinline__ float ex2w(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

enum WideBar : int {
  wKjFull = 0,  // the part's K columns (once)
  wQFull,       // Q, lse, delta of the step
  wQFree,       // dK of the step has read Q (and the dS pass lse / delta before it)
  wXKFull,      // the other K columns of the step, in X
  wXKFree,      // S^T has read them
  wDoFull,      // dO of the step, in X
  wXFree,       // dP^T and dV have read dO
  wBFull,       // bias tile of a query tile, in the bias / dS^T buffer
  wBDFree,      // dQ and dK of the step have read dS^T: the buffer is free
  wVFull,       // +slot (2): V chunk ring
  wVEmpty = wVFull + 2,
  wSFull = wVEmpty + 2,
  wPReady,   // P^T of the step stored in TMEM (compute threads)
  wDpFull,
  wDsReady,  // dS^T of the step stored in shared memory (compute threads)
  wDqFull,
  wDqFree,  // dQ read out of TMEM (drain threads)
  wFinal,
  wDrain,
  wNever,  // never arrived at: the target of the test wait (FDMA_FLAG_TEST_SHORT_WAIT)
  kNumWideBars
};

constexpr int kWideThreads = 512;
constexpr uint32_t kWRegsCtl = 48, kWRegsCompute = 160, kWRegsDrain = 144;
static_assert((kWRegsCtl + 2 * kWRegsCompute + kWRegsDrain) / 4 * kWideThreads <= 65536,
              "register split exceeds the register file");

template <int DQK, int DV, int KW>
struct WideSmem {
  static constexpr int kQC = DQK / 64;       // Q / K chunks of 64 columns (16 KB each)
  static constexpr int kVC = DV / 64;        // V / dO chunks
  static constexpr int kKjC = KW / 64;       // the part's K chunks
  static constexpr int kKoC = kQC - kKjC;    // the other K chunks
  static constexpr uint32_t kTail = 32768u + 1024u + kNumWideBars * 8u + 16u + kMaxKTiles / 4;
  // Resident plan, where it fits (192 / 128): all of K and all of V stay in shared memory for the
  // CTA's life and X holds only dO.  Otherwise (256 / 256) the part's K columns stay, X takes the
  // other K columns and then dO each step, and V streams through a two-slot ring of chunks.
  static constexpr bool kRes = (2u * kQC + 2u * kVC) * 16384u + kTail <= 232448u;
  static constexpr int kKC = kRes ? kQC : kKjC;  // K chunks kept (all, or the part's)
  static constexpr int kXC = kRes ? kVC : (kKoC > kVC ? kKoC : kVC);
  static constexpr int kVS = kRes ? kVC : 2;     // V chunks kept, or ring slots
  static constexpr uint32_t kOffQ = 0;
  static constexpr uint32_t kOffKj = kOffQ + kQC * 16384u;  // K: all chunks (resident) or the part's
  static constexpr uint32_t kOffX = kOffKj + kKC * 16384u;
  static constexpr uint32_t kOffV = kOffX + kXC * 16384u;
  static constexpr uint32_t kOffBD = kOffV + kVS * 16384u;  // bias tile / dS^T tile (32 KB)
  static constexpr uint32_t kOffLse = kOffBD + 32768u;
  static constexpr uint32_t kOffDelta = kOffLse + 512u;
  static constexpr uint32_t kOffBar = kOffDelta + 512u;
  static constexpr uint32_t kOffMisc = kOffBar + kNumWideBars * 8u;
  static constexpr uint32_t kOffMap = kOffMisc + 16u;  // this key tile's column of the block map, 2 bits per tile
  static constexpr uint32_t kTotal = kOffMap + kMaxKTiles / 4;
  static_assert(kTotal <= 232448u, "wide backward shared memory exceeds the per-CTA limit");
};

__host__ __device__ constexpr uint32_t wk_off(int k) {  // K-major step k of a 128-row tile of 64-column blocks
  return static_cast<uint32_t>(((k >> 2) * 128u * 128u + (k & 3) * 32u) >> 4);
}
__host__ __device__ constexpr uint32_t wmn_off(int k) { return static_cast<uint32_t>((k * 2048) >> 4); }

// Active query tiles of one key-tile column (2 bits per tile in shared memory).
struct WideCol {
  const uint8_t* map2;
  int nTq;
  __device__ __forceinline__ int cls(int qt) const { return (map2[qt >> 2] >> ((qt & 3) * 2)) & 3; }
  __device__ __forceinline__ int next(int qt) const {
    do {
      ++qt;
    } while (qt < nTq && cls(qt) == kSkip);
    return qt;
  }
  __device__ __forceinline__ int first() const { return next(-1); }
  __device__ __forceinline__ bool valid(int qt) const { return qt < nTq; }
};

template <int DQK, int DV, int PART, bool HAS_BIAS, bool WANT_DBIAS>
__global__ void __launch_bounds__(kWideThreads, 1)
    bwd_wide_kernel(const __grid_constant__ CUtensorMap tmQ, const __grid_constant__ CUtensorMap tmK,
                    const __grid_constant__ CUtensorMap tmV, const __grid_constant__ CUtensorMap tmDO,
                    const __grid_constant__ CUtensorMap tmB, const BwdParams p) {
  constexpr int KC0 = 128 * PART;  // first dK / dQ column of the part
  constexpr int KW = DQK - KC0 < 128 ? DQK - KC0 : 128;
  constexpr int VW = DV - KC0 <= 0 ? 0 : (DV - KC0 < 128 ? DV - KC0 : 128);
  static_assert(KW == 64 || KW == 128, "part widths are 64 or 128 columns");
  static_assert(VW == 0 || VW == 64 || VW == 128, "part widths are 64 or 128 columns");
  using L = WideSmem<DQK, DV, KW>;
  constexpr int QC = L::kQC, VC = L::kVC, KjC = L::kKjC, KoC = L::kKoC;
  constexpr bool RES = L::kRes;
  constexpr uint32_t IDESC_S = idesc_bf16(128, 128, false, false);            // S^T, dP^T
  constexpr uint32_t IDESC_DV = idesc_bf16(128, VW > 0 ? VW : 64, false, true);  // P^T(tmem) x dO part
  constexpr uint32_t IDESC_DK = idesc_bf16(128, KW, false, true);             // dS^T x Q part
  constexpr uint32_t IDESC_DQ = idesc_bf16(128, KW, true, true);              // dS (M contiguous) x K part

  extern __shared__ __align__(1024) uint8_t smem[];
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + L::kOffBar);
  uint32_t* misc = reinterpret_cast<uint32_t*>(smem + L::kOffMisc);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(misc + 1);
  uint8_t* sQ = smem + L::kOffQ;
  uint8_t* sKj = smem + L::kOffKj;
  uint8_t* sX = smem + L::kOffX;
  uint8_t* sV = smem + L::kOffV;
  uint8_t* sBD = smem + L::kOffBD;
  float* sLse = reinterpret_cast<float*>(smem + L::kOffLse);
  float* sDelta = reinterpret_cast<float*>(smem + L::kOffDelta);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  int id = blockIdx.x;
  const int g = id % p.Hkv;
  id /= p.Hkv;
  const int b = id % p.B;
  const int kt = id / p.B;  // small key tiles (most causal work) first
  const int k0 = kt * kTile;
  const int64_t col_base = static_cast<int64_t>(b * p.Hkv + g) * p.nTq * p.nTk + kt;
  uint8_t* map2 = smem + L::kOffMap;
  const WideCol it{map2, p.nTq};
  const bool ragged_k = (p.Nk & (kTile - 1)) != 0 && kt == p.nTk - 1;
  const bool ragged_q_any = (p.Nq & (kTile - 1)) != 0;

  if ((smem_u32(smem) & 1023u) != 0) {
    if (threadIdx.x == 0) atomicCAS(p.err, 0, kDevErrAlign);
    return;
  }
  if (threadIdx.x == 0) {
    for (int i = 0; i < kNumWideBars; ++i) mbar_init(&bars[i], 1);
    mbar_init(&bars[wPReady], 256);
    mbar_init(&bars[wDsReady], 256);
    mbar_init(&bars[wDqFree], 128);
    misc[1] = 0;
    fence_mbar_init();
  }
  for (int q = threadIdx.x; q < (p.nTq + 3) / 4; q += blockDim.x) {
    uint32_t v = 0;
    for (int e = 0; e < 4; ++e) {
      const int qt = 4 * q + e;
      if (qt < p.nTq) v |= static_cast<uint32_t>(p.kmap[col_base + static_cast<int64_t>(qt) * p.nTk] & 3) << (2 * e);
    }
    map2[q] = static_cast<uint8_t>(v);
  }
  if (warp == 1) {
    tmem_alloc(misc, 512);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tbase = misc[0];
  const int first_qt = it.first();
  const bool any_active = it.valid(first_qt);

  if (warp < 4) {
    regs_decrease<kWRegsCtl>();
    if (warp == 0 && lane == 0 && any_active) {
      // ------------------------------------------------------------ producer
      tma_prefetch_desc(&tmQ);
      tma_prefetch_desc(&tmK);
      tma_prefetch_desc(&tmV);
      tma_prefetch_desc(&tmDO);
      if (HAS_BIAS) tma_prefetch_desc(&tmB);
      if (RES) {  // all of K and V, once
        mbar_arrive_expect_tx(&bars[wKjFull], (QC + VC) * 16384u);
        for (int c = 0; c < QC; ++c) tma_load_4d(sKj + c * 16384, &tmK, &bars[wKjFull], c * 64, k0, g, b);
        for (int c = 0; c < VC; ++c) tma_load_4d(sV + c * 16384, &tmV, &bars[wKjFull], c * 64, k0, g, b);
      } else {
        mbar_arrive_expect_tx(&bars[wKjFull], KjC * 16384u);
        for (int c = 0; c < KjC; ++c) tma_load_4d(sKj + c * 16384, &tmK, &bars[wKjFull], KC0 + c * 64, k0, g, b);
      }
      int n = 0, nb = 0, nv = 0;      // steps, bias fills, V chunk fills issued
      int nq = 0, nxk = 0, ndo = 0;   // Q, other-K and dO fills issued
      bool ok = true;
      for (int qt = first_qt; ok && it.valid(qt); qt = it.next(qt)) {
        for (int hh = 0; hh < p.G; ++hh, ++n) {
          const int h = g * p.G + hh;
          // Q, lse and delta: the previous step's dK has read Q (its dS pass, before it, lse and delta)
          if (!(ok = mbar_wait(&bars[wQFree], (n & 1) ^ 1, p.err, kDevErrTimeout, abort_flag))) break;
          mbar_arrive_expect_tx(&bars[wQFull], QC * 16384u + 1024u);
          for (int c = 0; c < QC; ++c) tma_load_4d(sQ + c * 16384, &tmQ, &bars[wQFull], c * 64, qt * kTile, h, b);
          const int64_t vec = (static_cast<int64_t>(b) * p.Hq + h) * p.nqpad + qt * kTile;
          bulk_load(sLse, p.lse2 + vec, 512, &bars[wQFull]);
          bulk_load(sDelta, p.delta + vec, 512, &bars[wQFull]);
          nq = n + 1;
          // the other K columns, into X once the previous step's dP^T and dV have read dO there
          // (resident plan: X holds only dO)
          if (!(ok = mbar_wait(&bars[wXFree], (n & 1) ^ 1, p.err, kDevErrTimeout, abort_flag))) break;
          if (RES) {
          } else if (KoC > 0) {
            mbar_arrive_expect_tx(&bars[wXKFull], KoC * 16384u);
            for (int i = 0; i < KoC; ++i) {
              const int c = i < KC0 / 64 ? i : i + KjC;
              tma_load_4d(sX + i * 16384, &tmK, &bars[wXKFull], c * 64, k0, g, b);
            }
          } else {
            mbar_arrive(&bars[wXKFull]);
          }
          nxk = n + 1;
          // the query tile's bias, at its first head, once the previous step's dQ and dK have
          // read dS^T out of the buffer
          if (HAS_BIAS && hh == 0) {
            if (!(ok = mbar_wait(&bars[wBDFree], (n & 1) ^ 1, p.err, kDevErrTimeout, abort_flag))) break;
            mbar_arrive_expect_tx(&bars[wBFull], 32768u);
            for (int c = 0; c < 2; ++c)
              tma_load_4d(sBD + c * 16384, &tmB, &bars[wBFull], k0 + c * 64, qt * kTile, g * p.bias_hsel,
                          b * p.bias_bsel);
            ++nb;
          }
          // dO, into X once S^T has read the other K columns
          if (!RES && !(ok = mbar_wait(&bars[wXKFree], n & 1, p.err, kDevErrTimeout, abort_flag))) break;
          mbar_arrive_expect_tx(&bars[wDoFull], VC * 16384u);
          for (int c = 0; c < VC; ++c) tma_load_4d(sX + c * 16384, &tmDO, &bars[wDoFull], c * 64, qt * kTile, h, b);
          ndo = n + 1;
          // V, in 64-column chunks through the two-slot ring (resident plan: loaded once)
          for (int c = 0; !RES && ok && c < VC; ++c, ++nv) {
            const int s = nv & 1;
            if (!(ok = mbar_wait(&bars[wVEmpty + s], ((nv >> 1) & 1) ^ 1, p.err, kDevErrTimeout, abort_flag))) break;
            mbar_arrive_expect_tx(&bars[wVFull + s], 16384u);
            tma_load_4d(sV + s * 16384, &tmV, &bars[wVFull + s], c * 64, k0, g, b);
          }
          if (!ok) break;
        }
      }
      if (*abort_flag) {
        // let this CTA's own copies land before it retires (bounded waits): only the last fill
        // of each buffer (of each ring slot) can still be in flight
        mbar_wait(&bars[wKjFull], 0, p.err, kDevErrTimeout, nullptr);
        if (nq > 0) mbar_wait(&bars[wQFull], (nq - 1) & 1, p.err, kDevErrTimeout, nullptr);
        if (!RES && nxk > 0) mbar_wait(&bars[wXKFull], (nxk - 1) & 1, p.err, kDevErrTimeout, nullptr);
        if (ndo > 0) mbar_wait(&bars[wDoFull], (ndo - 1) & 1, p.err, kDevErrTimeout, nullptr);
        if (nb > 0) mbar_wait(&bars[wBFull], (nb - 1) & 1, p.err, kDevErrTimeout, nullptr);
        for (int m = nv > 2 ? nv - 2 : 0; m < nv; ++m)
          mbar_wait(&bars[wVFull + (m & 1)], (m >> 1) & 1, p.err, kDevErrTimeout, nullptr);
      }
    } else if (warp == 1 && lane == 0 && any_active) {
      // ------------------------------------------------------------ MMA issuer
      bool ok = mbar_wait(&bars[wKjFull], 0, p.err, kDevErrTimeout, abort_flag);
      const uint64_t dsdesc_k = sdesc_sw128(smem_u32(sBD), 16, 1024);
      const uint64_t dsdesc_mn = sdesc_sw128(smem_u32(sBD), 16384, 1024);
      const uint64_t kjdesc_mn = sdesc_sw128(smem_u32(sKj + (RES ? (KC0 / 64) * 16384 : 0)), 16384, 1024);
      const uint64_t qdesc_mn = sdesc_sw128(smem_u32(sQ + (KC0 / 64) * 16384), 16384, 1024);
      const uint64_t dodesc_mn = sdesc_sw128(smem_u32(sX + (KC0 / 64) * 16384), 16384, 1024);
      int n = 0, nv = 0;
      for (int qt = first_qt; ok && it.valid(qt); qt = it.next(qt)) {
        for (int hh = 0; hh < p.G; ++hh, ++n) {
          // S^T = K Q^T over the full q/k width: the part's chunks from their resident copy,
          // the others from X
          if (!(ok = mbar_wait(&bars[wQFull], n & 1, p.err, kDevErrTimeout, abort_flag) &&
                     (RES || mbar_wait(&bars[wXKFull], n & 1, p.err, kDevErrTimeout, abort_flag))))
            break;
          tc_fence_after();
          for (int c = 0; c < QC; ++c) {
            const bool own = c >= KC0 / 64 && c < KC0 / 64 + KjC;
            const uint8_t* ka = RES ? sKj + c * 16384
                                    : own ? sKj + (c - KC0 / 64) * 16384 : sX + (c < KC0 / 64 ? c : c - KjC) * 16384;
            const uint64_t adesc = sdesc_sw128(smem_u32(ka), 16, 1024);
            const uint64_t bdesc = sdesc_sw128(smem_u32(sQ + c * 16384), 16, 1024);
            const uint32_t acc0 = c > 0 ? 1u : 0u;
            umma_ss_off<wk_off(0), wk_off(0)>(tbase, adesc, bdesc, IDESC_S, acc0);
            umma_ss_off<wk_off(1), wk_off(1)>(tbase, adesc, bdesc, IDESC_S, 1u);
            umma_ss_off<wk_off(2), wk_off(2)>(tbase, adesc, bdesc, IDESC_S, 1u);
            umma_ss_off<wk_off(3), wk_off(3)>(tbase, adesc, bdesc, IDESC_S, 1u);
          }
          umma_commit(&bars[wSFull]);
          if (!RES) umma_commit(&bars[wXKFree]);
          // dP^T = V dO^T over the full v width into columns 128..255, which the previous
          // step's dQ used
          if (!(ok = mbar_wait(&bars[wDoFull], n & 1, p.err, kDevErrTimeout, abort_flag))) break;
          if (n > 0 && !(ok = mbar_wait(&bars[wDqFree], (n - 1) & 1, p.err, kDevErrTimeout, abort_flag))) break;
          for (int c = 0; c < VC; ++c, ++nv) {
            const int s = RES ? c : (nv & 1);  // resident V chunk c, or ring slot
            if (!RES && !(ok = mbar_wait(&bars[wVFull + s], (nv >> 1) & 1, p.err, kDevErrTimeout, abort_flag))) break;
            tc_fence_after();
            const uint64_t adesc = sdesc_sw128(smem_u32(sV + s * 16384), 16, 1024);
            const uint64_t bdesc = sdesc_sw128(smem_u32(sX + c * 16384), 16, 1024);
            const uint32_t acc0 = c > 0 ? 1u : 0u;
            umma_ss_off<wk_off(0), wk_off(0)>(tbase + 128, adesc, bdesc, IDESC_S, acc0);
            umma_ss_off<wk_off(1), wk_off(1)>(tbase + 128, adesc, bdesc, IDESC_S, 1u);
            umma_ss_off<wk_off(2), wk_off(2)>(tbase + 128, adesc, bdesc, IDESC_S, 1u);
            umma_ss_off<wk_off(3), wk_off(3)>(tbase + 128, adesc, bdesc, IDESC_S, 1u);
            if (!RES) umma_commit(&bars[wVEmpty + s]);
          }
          if (!ok) break;
          umma_commit(&bars[wDpFull]);
          // dV += P^T dO  (the part's dO columns; K dimension = 128 queries; P^T packed in TMEM
          // columns 0..31 and 64..95)
          if (!(ok = mbar_wait(&bars[wPReady], n & 1, p.err, kDevErrTimeout, abort_flag))) break;
          tc_fence_after();
          if (VW > 0) {
            static_for<0, 8>([&](auto kc) {
              constexpr int k = decltype(kc)::value;
              umma_ts_off<k * 8 + (k >= 4 ? 32 : 0), wmn_off(k)>(tbase + 256, tbase, dodesc_mn, IDESC_DV,
                                                                 (n > 0 || k > 0) ? 1u : 0u);
            });
          }
          umma_commit(&bars[wXFree]);  // dP^T and dV have read dO
          // dQ = dS K (the part's columns) over columns 128.., then dK += dS^T Q (the part's columns)
          if (!(ok = mbar_wait(&bars[wDsReady], n & 1, p.err, kDevErrTimeout, abort_flag))) break;
          tc_fence_after();
          static_for<0, 8>([&](auto kc) {
            constexpr int k = decltype(kc)::value;
            umma_ss_off<wmn_off(k), wmn_off(k)>(tbase + 128, dsdesc_mn, kjdesc_mn, IDESC_DQ, k > 0 ? 1u : 0u);
          });
          umma_commit(&bars[wDqFull]);
          static_for<0, 8>([&](auto kc) {
            constexpr int k = decltype(kc)::value;
            umma_ss_off<wk_off(k), wmn_off(k)>(tbase + 384, dsdesc_k, qdesc_mn, IDESC_DK, (n > 0 || k > 0) ? 1u : 0u);
          });
          umma_commit(&bars[wQFree]);
          umma_commit(&bars[wBDFree]);
        }
      }
      umma_commit(&bars[wFinal]);
      umma_commit(&bars[wDrain]);
      mbar_wait(&bars[wDrain], 0, p.err, kDevErrTimeout, nullptr);
    }
  } else if (warp < 12) {
    regs_increase<kWRegsCompute>();
    // ------------------------------------------------------------ compute
    // Warpgroup wg owns queries 64*wg .. 64*wg+63 of every step; thread (quad, lane) owns key
    // row j of S^T / dP^T / dK / dV.
    const int wg = (warp - 4) >> 2;
    const int quad = warp & 3;
    const int j = quad * 32 + lane;
    const int ctid = (warp - 4) * 32 + lane;  // 0..255
    const int kidx = k0 + j;
    const bool kin = kidx < p.Nk;
    const uint32_t tl = tbase + (static_cast<uint32_t>(quad * 32) << 16);
    const int qbase = wg * 64;
    uint64_t acc2[WANT_DBIAS ? 32 : 1];  // dBias partial sums (of scale * dS), pairs of queries
#pragma unroll
    for (int c = 0; c < (WANT_DBIAS ? 32 : 1); ++c) acc2[c] = 0ull;
    const uint64_t sc2 = f2(p.scale_log2, p.scale_log2);
    const uint64_t scl2 = f2(p.scale, p.scale);
    const uint64_t lg2 = f2(kLog2eW, kLog2eW);
    int n = 0, qi = 0;
    bool ok = !p.test_short_wait || mbar_wait(&bars[wNever], 0, p.err, kDevErrTimeout, abort_flag, kTestWaitNs);
    // No compute thread leaves these loops early, so every one of them reaches every named
    // barrier; after a failed wait (ok == false) the work and the stores are skipped.
    uint32_t bw0 = ~0u, bw1 = ~0u;
    uint32_t bpk[HAS_BIAS ? 32 : 1];
    auto store_dbias = [&](int q0t) {
      const uint64_t inv2 = f2(1.f / p.scale, 1.f / p.scale);  // the sums are of scale * dS
      const bool odd = (j & 1) != 0;
      const int col = kidx & ~1;
      uint32_t* base = reinterpret_cast<uint32_t*>(
          p.dbias + ((static_cast<int64_t>(b) * p.Hkv + g) * p.Nq + q0t + qbase + (odd ? 1 : 0)) * p.Nk + col);
#pragma unroll
      for (int qp = 0; qp < 32; ++qp) {
        float a0, a1;
        f2split(mul2(acc2[qp], inv2), a0, a1);
        const uint32_t w = pack_bf16x2(a0, a1);  // (query 2qp, query 2qp+1) of key j
        const uint32_t send = odd ? (w & 0xFFFFu) : (w >> 16);
        const uint32_t got = __shfl_xor_sync(0xffffffffu, send, 1);
        const uint32_t pair = odd ? (got | (w & 0xFFFF0000u)) : ((w & 0xFFFFu) | (got << 16));
        const int row = q0t + qbase + 2 * qp + (odd ? 1 : 0);
        if (ok && row < p.Nq && kin) base[static_cast<int64_t>(qp) * p.Nk] = pair;
        acc2[qp] = 0ull;
      }
    };
    int q0_prev = 0;
    for (int qt = first_qt; it.valid(qt); qt = it.next(qt), ++qi) {
      const int q0 = qt * kTile;
      if (WANT_DBIAS && qi > 0) store_dbias(q0_prev);
      // the tile's keep bits and bias^T slice, into registers (the bias buffer then takes dS^T)
      {
        uint2 bb = make_uint2(~0u, ~0u);
        if (it.cls(qt) == kPartial || ragged_k || (ragged_q_any && qt == p.nTq - 1)) {
          const int64_t tile = col_base + static_cast<int64_t>(qt) * p.nTk;
          bb = reinterpret_cast<const uint2*>(&p.bits_col[tile * kTile + j])[wg];
        }
        bw0 = bb.x;
        bw1 = bb.y;
      }
      if (HAS_BIAS) {
        ok = ok && mbar_wait(&bars[wBFull], qi & 1, p.err, kDevErrTimeout, abort_flag);
        if (ok) {
          const uint8_t* bt = sBD + (j >> 6) * 16384 + (j & 7) * 2;
          const int jc = (j & 63) >> 3;
#pragma unroll
          for (int e = 0; e < 32; ++e) {
            const int i0 = qbase + 2 * e, i1 = i0 + 1;
            const uint32_t lo = *reinterpret_cast<const uint16_t*>(bt + i0 * 128 + ((jc ^ (i0 & 7)) << 4));
            const uint32_t hi = *reinterpret_cast<const uint16_t*>(bt + i1 * 128 + ((jc ^ (i1 & 7)) << 4));
            // masked pairs get a bias of -inf (bf16 0xFF80): their P is exp2(-inf) = 0
            const uint32_t wd = e < 16 ? bw0 : bw1;
            const bool k0b = (wd >> ((2 * e) & 31)) & 1u, k1b = (wd >> ((2 * e + 1) & 31)) & 1u;
            bpk[e] = (k0b ? lo : 0xFF80u) | ((k1b ? hi : 0xFF80u) << 16);
          }
        }
        // the buffer is next written by this step's dS^T stores (all compute threads must have
        // read the bias first) and later by TMA (the proxy fence orders these reads before it)
        fence_proxy_async_smem();
        named_bar_sync(1, 256);
      }
      for (int hh = 0; hh < p.G; ++hh, ++n) {
        // ---------------- P pass: P^T = exp2(S^T * scale*log2e + bias^T*log2e - lse*log2e)
        ok = ok && mbar_wait(&bars[wSFull], n & 1, p.err, kDevErrTimeout, abort_flag);
        ok = ok && mbar_wait(&bars[wQFull], n & 1, p.err, kDevErrTimeout, abort_flag);
        if (ok) {
          tc_fence_after();
          const float* lse2 = sLse + qbase;
#pragma unroll
          for (int c = 0; c < 4; ++c) {  // 16 queries per chunk
            const int col = qbase + c * 16;
            uint32_t sr[16];
            tmem_ld16(tl + col, sr);
            uint64_t nl[8];
#pragma unroll
            for (int v = 0; v < 4; ++v) {
              const ulonglong2 a = reinterpret_cast<const ulonglong2*>(lse2 + c * 16)[v];
              nl[2 * v] = a.x;
              nl[2 * v + 1] = a.y;
            }
            tmem_ld_wait(sr);
            const uint32_t word = c < 2 ? bw0 : bw1;
            uint32_t pk[8];
#pragma unroll
            for (int e = 0; e < 16; e += 2) {
              const int qq = c * 16 + e;
              const uint64_t s2 = f2(__uint_as_float(sr[e]), __uint_as_float(sr[e + 1]));
              const uint64_t x2 = HAS_BIAS ? fma2(s2, sc2, fma2(bf16x2_to_f2(bpk[qq >> 1]), lg2, nl[e >> 1]))
                                           : fma2(s2, sc2, nl[e >> 1]);
              float x0, x1;
              f2split(x2, x0, x1);
              const float p0 = (HAS_BIAS || ((word >> (qq & 31)) & 1u)) ? ex2w(x0) : 0.f;
              const float p1 = (HAS_BIAS || ((word >> ((qq + 1) & 31)) & 1u)) ? ex2w(x1) : 0.f;
              pk[e >> 1] = pack_bf16x2(p0, p1);
            }
            tmem_st8(tl + wg * 64 + c * 8, pk);  // queries 0..63 -> cols 0..31, 64..127 -> 64..95
          }
          tmem_st_wait();
          tc_fence_before();
          mbar_arrive(&bars[wPReady]);
        }
        // ---------------- dS pass: scale * dS^T = P^T (scale * dP^T - scale * delta)
        ok = ok && mbar_wait(&bars[wDpFull], n & 1, p.err, kDevErrTimeout, abort_flag);
        // the previous step's dQ and dK have read the dS^T tile
        ok = ok && (n == 0 || mbar_wait(&bars[wBDFree], (n - 1) & 1, p.err, kDevErrTimeout, abort_flag));
        if (ok) {
          tc_fence_after();
          const float* dlt = sDelta + qbase;
#pragma unroll
          for (int c = 0; c < 4; ++c) {
            const int col = qbase + c * 16;
            uint32_t pp[8], dr[16];
            tmem_ld8(tl + wg * 64 + c * 8, pp);
            tmem_ld16(tl + 128 + col, dr);
            uint64_t dd[8];
#pragma unroll
            for (int v = 0; v < 4; ++v) {
              const ulonglong2 bq = reinterpret_cast<const ulonglong2*>(dlt + c * 16)[v];
              dd[2 * v] = bq.x;
              dd[2 * v + 1] = bq.y;
            }
            tmem_ld_wait(dr);
            tmem_ld_tie(pp);
            uint32_t dk[8];
#pragma unroll
            for (int e = 0; e < 16; e += 2) {
              const int qq = c * 16 + e;
              const uint64_t dv2 = mul2(bf16x2_to_f2(pp[e >> 1]),
                                        fma2(f2(__uint_as_float(dr[e]), __uint_as_float(dr[e + 1])), scl2, dd[e >> 1]));
              if (WANT_DBIAS) acc2[qq >> 1] = add2(acc2[qq >> 1], dv2);
              float d0, d1;
              f2split(dv2, d0, d1);
              dk[e >> 1] = pack_bf16x2(d0, d1);
            }
            // dS^T row j, queries col..col+15: two 16-byte chunks of the SW128 K-major tile
            uint8_t* rowp = sBD + wg * 16384 + j * 128;
            *reinterpret_cast<uint4*>(rowp + (((2 * c) ^ (j & 7)) << 4)) = make_uint4(dk[0], dk[1], dk[2], dk[3]);
            *reinterpret_cast<uint4*>(rowp + (((2 * c + 1) ^ (j & 7)) << 4)) = make_uint4(dk[4], dk[5], dk[6], dk[7]);
          }
          fence_proxy_async_smem();
          tc_fence_before();
          mbar_arrive(&bars[wDsReady]);
        }
      }
      q0_prev = q0;
    }
    if (WANT_DBIAS && n > 0) store_dbias(q0_prev);
    if (ok && n > 0) ok = mbar_wait(&bars[wFinal], 0, p.err, kDevErrTimeout, abort_flag);
    // zero-fill the dBias tiles of this key column that were skipped: 16 bytes per thread and
    // row (Nk is a multiple of 8: a chunk is all in or all out)
    if (WANT_DBIAS && ok) {
      const int ch = ctid & 15, r0 = ctid >> 4;
      const int c = k0 + ch * 8;
      if (c < p.Nk) {
        const int64_t step = static_cast<int64_t>(p.Nk) * 2;  // 16 rows, in 16-byte units
        for (int qt = 0; qt < p.nTq; ++qt) {
          if (it.cls(qt) != kSkip) continue;
          const int rows = min(kTile, p.Nq - qt * kTile);
          uint4* dst = reinterpret_cast<uint4*>(
              p.dbias + ((static_cast<int64_t>(b) * p.Hkv + g) * p.Nq + qt * kTile + r0) * p.Nk + c);
          for (int r = r0; r < rows; r += 16, dst += step) *dst = make_uint4(0u, 0u, 0u, 0u);
        }
      }
    }
    // the part's dK columns (warpgroup 0) and dV columns (warpgroup 1); both carry their scale
    if (ok && (wg == 0 || VW > 0)) {
      tc_fence_after();
      const int W = wg == 0 ? KW : VW;
      uint16_t* dst = wg == 0 ? p.dk + ((static_cast<int64_t>(b) * p.Nk + kidx) * p.Hkv + g) * DQK + KC0
                              : p.dv + ((static_cast<int64_t>(b) * p.Nk + kidx) * p.Hkv + g) * DV + KC0;
      const uint32_t col0 = wg == 0 ? 384u : 256u;
      for (int c = 0; c < W / 32; ++c) {
        uint32_t r[32];
        if (n > 0) {
          tmem_ld32(tl + col0 + c * 32, r);
          tmem_ld_wait(r);
        } else {
#pragma unroll
          for (int t = 0; t < 32; ++t) r[t] = 0u;
        }
        uint32_t pk[16];
#pragma unroll
        for (int t = 0; t < 16; ++t) pk[t] = pack_bf16x2(__uint_as_float(r[2 * t]), __uint_as_float(r[2 * t + 1]));
        if (kin) {
          uint4* d4 = reinterpret_cast<uint4*>(dst + c * 32);
#pragma unroll
          for (int v = 0; v < 4; ++v) d4[v] = make_uint4(pk[4 * v], pk[4 * v + 1], pk[4 * v + 2], pk[4 * v + 3]);
        }
      }
    }
  } else {
    regs_increase<kWRegsDrain>();
    if (any_active) {
      // ------------------------------------------------------------ dQ drain
      // Warp (12 + quad) reads TMEM lanes quad*32..+31 (queries) of each step's dQ part, frees
      // the columns for the next dP^T and adds the rows to the fp32 accumulator.
      const int quad = warp & 3;
      const int row = quad * 32 + lane;
      const uint32_t tl = tbase + (static_cast<uint32_t>(quad * 32) << 16);
      int n = 0;
      bool ok = true;
      for (int qt = first_qt; ok && it.valid(qt); qt = it.next(qt)) {
        const int i = qt * kTile + row;
        for (int hh = 0; hh < p.G; ++hh, ++n) {
          const int h = g * p.G + hh;
          if (!(ok = mbar_wait(&bars[wDqFull], n & 1, p.err, kDevErrTimeout, abort_flag))) break;
          tc_fence_after();
          uint32_t r[KW / 32][32];
#pragma unroll
          for (int c = 0; c < KW / 32; ++c) tmem_ld32(tl + 128 + c * 32, r[c]);
          tmem_ld_wait(r[0]);
#pragma unroll
          for (int c = 1; c < KW / 32; ++c) tmem_ld_tie(r[c]);
          tc_fence_before();
          mbar_arrive(&bars[wDqFree]);
          if (i < p.Nq) {
            // the accumulator is grouped by four head-dim columns: a warp's reductions of one
            // group cover 32 consecutive queries, 512 contiguous bytes
            float* dst = p.dq_acc + dq_acc_index(b, h, i, KC0, p.Hq, p.nqpad, DQK);
            const int64_t gstep = static_cast<int64_t>(p.nqpad) * 4;  // next group of four columns
#pragma unroll
            for (int c = 0; c < KW / 32; ++c)
#pragma unroll
              for (int v = 0; v < 8; ++v)
                red_add_v4(dst + (c * 8 + v) * gstep, __uint_as_float(r[c][4 * v]), __uint_as_float(r[c][4 * v + 1]),
                           __uint_as_float(r[c][4 * v + 2]), __uint_as_float(r[c][4 * v + 3]));
          }
        }
      }
    }
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    __syncwarp();
    tc_fence_after();
    tmem_dealloc(tbase, 512);
  }
}

template <int DQK, int DV, int PART, bool HB, bool WD>
cudaError_t launch_wide_t(const CUtensorMap& tq, const CUtensorMap& tk, const CUtensorMap& tv,
                          const CUtensorMap& tdo, const CUtensorMap& tb, const BwdParams& p, cudaStream_t stream) {
  constexpr int KW = DQK - 128 * PART < 128 ? DQK - 128 * PART : 128;
  using L = WideSmem<DQK, DV, KW>;
  auto kern = bwd_wide_kernel<DQK, DV, PART, HB, WD>;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, L::kTotal);
  if (e != cudaSuccess) return e;
  cudaFuncAttributes fa;
  e = cudaFuncGetAttributes(&fa, kern);
  if (e != cudaSuccess) return e;
  // the setmaxnreg split needs the launch allocation to cover it
  if (fa.numRegs < static_cast<int>((kWRegsCtl + 2 * kWRegsCompute + kWRegsDrain) / 4))
    return cudaErrorInvalidConfiguration;
  const unsigned grid = static_cast<unsigned>(p.nTk) * p.B * p.Hkv;
  kern<<<grid, kWideThreads, L::kTotal, stream>>>(tq, tk, tv, tdo, tb, p);
  return cudaGetLastError();
}

// Both parts; dBias (when wanted) is formed by part 0 only.
template <int DQK, int DV, bool HB>
cudaError_t launch_wide_parts(bool want_dbias, const CUtensorMap& tq, const CUtensorMap& tk, const CUtensorMap& tv,
                              const CUtensorMap& tdo, const CUtensorMap& tb, const BwdParams& p,
                              cudaStream_t stream) {
  cudaError_t e = (HB && want_dbias) ? launch_wide_t<DQK, DV, 0, HB, HB>(tq, tk, tv, tdo, tb, p, stream)
                                     : launch_wide_t<DQK, DV, 0, HB, false>(tq, tk, tv, tdo, tb, p, stream);
  if (e != cudaSuccess) return e;
  return launch_wide_t<DQK, DV, 1, HB, false>(tq, tk, tv, tdo, tb, p, stream);
}

}  // namespace

cudaError_t launch_bwd_wide(int d, int dv, bool has_bias, bool want_dbias, const CUtensorMap& tq,
                            const CUtensorMap& tk, const CUtensorMap& tv, const CUtensorMap& tdo,
                            const CUtensorMap& tb, const BwdParams& p, cudaStream_t stream) {
  if (d == 192 && dv == 128)
    return has_bias ? launch_wide_parts<192, 128, true>(want_dbias, tq, tk, tv, tdo, tb, p, stream)
                    : launch_wide_parts<192, 128, false>(false, tq, tk, tv, tdo, tb, p, stream);
  if (d == 256 && dv == 256)
    return has_bias ? launch_wide_parts<256, 256, true>(want_dbias, tq, tk, tv, tdo, tb, p, stream)
                    : launch_wide_parts<256, 256, false>(false, tq, tk, tv, tdo, tb, p, stream);
  return cudaErrorInvalidValue;
}

}  // namespace fdma
