// Forward kernel: tiled attention with dynamic mask and learnable bias
// (Flash-DMA issue #73, "Project Progress": masked entries become -inf, the
// scale applies to QK^T, the bias is added, softmax, then P V; Flash-DMA
// README, "Key Features": blocks whose mask OR is false are skipped with no
// K/V/bias traffic; FlashMask README, "Sparse computation": element-wise
// masking only on partially masked blocks).
//
// One CTA = one (batch, query head, 128-row query tile).  Six warps:
//   warp 0      TMA producer: Q once, then K, V and the 128x128 bias tile of
//               every ACTIVE key tile into rings (skipped tiles are never
//               requested): two slots each, or one where a 192- or 256-wide
//               tile leaves no room for two in shared memory;
//   warp 1      TMEM owner and single-thread tcgen05.mma issuer:
//               S_n = Q K_n^T (SS, fp32 in TMEM, double-buffered), then
//               O += P_{n-1} V_{n-1} with P read from TMEM (TS);
//   warps 2..5  softmax, one thread per query row (TMEM lane): while S is
//               computed, the tile's additive term (bias, -inf at masked keys)
//               is formed from the bias tile and the keep bits; then S is
//               added with paired fp32 FMAs, a three-input row maximum, lazy O
//               rescaling, exp2 and P written back to TMEM as packed bf16 with
//               the row sum of the rounded weights; final O / l and lse.
// TMEM columns: S[0] 0..127, S[1] 128..255, O 256..256+dv.
// This one-head kernel serves the wide head dims, q/k width DQK and v/out width DV
// of 192 / 128 and 256 / 256 (FlashMask README, "Performance", SM100 head-dim
// table); head dims up to 128 run on the two-slot kernel further down.
#include "fdma_internal.h"
#include "fdma_ptx.cuh"

namespace fdma {
namespace {

constexpr float kLog2e = 1.4426950408889634f;
constexpr float kLn2 = 0.6931471805599453f;
constexpr float kRescaleThreshold = 8.0f;  // log2 units: P stays <= 2^8 between rescales
#define kNegInf (-__int_as_float(0x7f800000))

__device__ __forceinline__ float ex2(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

enum FwdBar : int {
  kQFull = 0,
  kKFull = 1,    // +slot
  kKEmpty = 3,   // +slot
  kVFull = 5,    // +slot
  kVEmpty = 7,   // +slot
  kBFull = 9,    // +slot
  kBEmpty = 11,  // +slot
  kSFull = 13,   // +slot
  kPReady = 15,  // +slot
  kODone = 17,
  kOFinal = 18,
  kDrain = 19,
  kFNever = 20,  // never arrived at: the target of the test wait (FDMA_FLAG_TEST_SHORT_WAIT)
  kNumFwdBars = 21
};

template <int DQK, int DV, bool HAS_BIAS>
struct FwdSmem {
  static constexpr uint32_t kQB = 128u * DQK * 2u;  // one Q or K tile (bf16)
  static constexpr uint32_t kVB = 128u * DV * 2u;   // one V tile
  static constexpr uint32_t kBB = 128u * 128u * 2u;
  static constexpr int kKS = DQK <= 128 ? 2 : 1;  // K ring slots
  static constexpr int kVS = DV <= 128 ? 2 : 1;   // V ring slots
  static constexpr uint32_t kOffQ = 0;
  static constexpr uint32_t kOffK = kQB;
  static constexpr uint32_t kOffV = kOffK + kKS * kQB;
  static constexpr uint32_t kOffBias = kOffV + kVS * kVB;
  static constexpr uint32_t kTail = kNumFwdBars * 8 + kMaxKTiles + 16;  // barriers, map row, misc
  // bias ring slots: two where they fit in the 227 KB a CTA may use, else one
  static constexpr int kBS = !HAS_BIAS ? 0 : (kOffBias + 2 * kBB + kTail <= 232448u ? 2 : 1);
  static constexpr int kBSlots = kBS > 0 ? kBS : 1;  // (for slot arithmetic without a bias)
  static constexpr uint32_t kOffBar = kOffBias + kBS * kBB;
  static constexpr uint32_t kOffMap = kOffBar + kNumFwdBars * 8;
  static constexpr uint32_t kOffMisc = kOffMap + kMaxKTiles;
  static constexpr uint32_t kTotal = kOffMisc + 16;
  static_assert(kTotal <= 232448u, "forward shared memory exceeds the per-CTA limit");
};

__device__ __forceinline__ int next_active(const int8_t* row, int kt, int n) {
  do {
    ++kt;
  } while (kt < n && row[kt] == kSkip);
  return kt;
}

// Descriptor offset (in the 16-byte units of the start-address field) of the
// k-th 16-element K step inside a K-major SW128 tile made of 64-column blocks.
__device__ __forceinline__ uint64_t kmajor_step(int k, uint32_t rows) {
  return static_cast<uint64_t>(((k >> 2) * rows * 128u + (k & 3) * 32u) >> 4);
}

template <int DQK, int DV, bool HAS_BIAS>
__global__ void __launch_bounds__(192, 1)
    fwd_kernel(const __grid_constant__ CUtensorMap tmQ, const __grid_constant__ CUtensorMap tmK,
               const __grid_constant__ CUtensorMap tmV, const __grid_constant__ CUtensorMap tmB,
               const FwdParams p) {
  using L = FwdSmem<DQK, DV, HAS_BIAS>;
  constexpr int KB = DQK / 64;  // 64-column swizzle blocks along the q/k head dim
  constexpr int VB = DV / 64;   // ... along the v head dim
  constexpr int KS = L::kKS, VS = L::kVS, BS = L::kBSlots;
  constexpr uint32_t IDESC_S = idesc_bf16(128, 128, false, false);
  constexpr uint32_t IDESC_O = idesc_bf16(128, DV, false, true);

  extern __shared__ __align__(1024) uint8_t smem[];
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + L::kOffBar);
  int8_t* map_row = reinterpret_cast<int8_t*>(smem + L::kOffMap);
  uint32_t* misc = reinterpret_cast<uint32_t*>(smem + L::kOffMisc);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(misc + 1);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  int id = blockIdx.x;
  const int hh = id % p.G;
  id /= p.G;
  const int g = id % p.Hkv;
  id /= p.Hkv;
  const int b = id % p.B;
  id /= p.B;
  const int qt = p.nTq - 1 - id;  // longest causal rows first
  const int h = g * p.G + hh;
  const int q0 = qt * kTile;
  const int64_t tile_base = (static_cast<int64_t>(b * p.Hkv + g) * p.nTq + qt) * p.nTk;
  const bool ragged_k = (p.Nk & (kTile - 1)) != 0;

  if ((smem_u32(smem) & 1023u) != 0) {
    if (threadIdx.x == 0) atomicCAS(p.err, 0, kDevErrAlign);
    return;
  }
  if (threadIdx.x == 0) {
    for (int i = 0; i < kNumFwdBars; ++i) mbar_init(&bars[i], 1);
    mbar_init(&bars[kBEmpty + 0], 128);
    mbar_init(&bars[kBEmpty + 1], 128);
    mbar_init(&bars[kPReady + 0], 128);
    mbar_init(&bars[kPReady + 1], 128);
    misc[1] = 0;
    fence_mbar_init();
  }
  for (int kt = threadIdx.x; kt < p.nTk; kt += blockDim.x) map_row[kt] = p.kmap[tile_base + kt];
  if (warp == 1) {
    tmem_alloc(misc, 512);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tbase = misc[0];
  const int first_kt = next_active(map_row, -1, p.nTk);
  const bool any_active = first_kt < p.nTk;

  uint8_t* sQ = smem + L::kOffQ;
  uint8_t* sK = smem + L::kOffK;
  uint8_t* sV = smem + L::kOffV;
  uint8_t* sB = smem + L::kOffBias;

  if (warp == 0) {
    // ------------------------------------------------------------ producer
    if (lane == 0 && any_active) {
      tma_prefetch_desc(&tmQ);
      tma_prefetch_desc(&tmK);
      tma_prefetch_desc(&tmV);
      if (HAS_BIAS) tma_prefetch_desc(&tmB);
      const uint64_t bias_pol = l2_evict_first();  // each bias tile is read once
      mbar_arrive_expect_tx(&bars[kQFull], L::kQB);
#pragma unroll
      for (int c = 0; c < KB; ++c) tma_load_4d(sQ + c * 16384, &tmQ, &bars[kQFull], c * 64, q0, h, b);
      int n = 0;
      int nk = 0, nb = 0, nv = 0;  // fills issued into the K, bias and V rings
      for (int kt = first_kt; kt < p.nTk; kt = next_active(map_row, kt, p.nTk), ++n) {
        const int k0 = kt * kTile;
        const int sk = n % KS, sb = n % BS, sv = n % VS;
        if (!mbar_wait(&bars[kKEmpty + sk], ((n / KS) & 1) ^ 1, p.err, kDevErrTimeout, abort_flag)) break;
        mbar_arrive_expect_tx(&bars[kKFull + sk], L::kQB);
#pragma unroll
        for (int c = 0; c < KB; ++c)
          tma_load_4d(sK + sk * L::kQB + c * 16384, &tmK, &bars[kKFull + sk], c * 64, k0, g, b);
        nk = n + 1;
        if (HAS_BIAS) {
          if (!mbar_wait(&bars[kBEmpty + sb], ((n / BS) & 1) ^ 1, p.err, kDevErrTimeout, abort_flag)) break;
          mbar_arrive_expect_tx(&bars[kBFull + sb], L::kBB);
#pragma unroll
          for (int c = 0; c < 2; ++c)
            tma_load_4d_hint(sB + sb * L::kBB + c * 16384, &tmB, &bars[kBFull + sb], k0 + c * 64, q0,
                             g * p.bias_hsel, b * p.bias_bsel, bias_pol);
          nb = n + 1;
        }
        if (!mbar_wait(&bars[kVEmpty + sv], ((n / VS) & 1) ^ 1, p.err, kDevErrTimeout, abort_flag)) break;
        mbar_arrive_expect_tx(&bars[kVFull + sv], L::kVB);
#pragma unroll
        for (int c = 0; c < VB; ++c)
          tma_load_4d(sV + sv * L::kVB + c * 16384, &tmV, &bars[kVFull + sv], c * 64, k0, g, b);
        nv = n + 1;
      }
      if (*abort_flag) {
        // let our own copies land before the CTA retires: in each ring only the last fill
        // of every slot can still be in flight (earlier ones were consumed before the slot
        // was refilled)
        mbar_wait(&bars[kQFull], 0, p.err, kDevErrTimeout, nullptr);
        for (int m = nk > KS ? nk - KS : 0; m < nk; ++m)
          mbar_wait(&bars[kKFull + m % KS], (m / KS) & 1, p.err, kDevErrTimeout, nullptr);
        for (int m = nv > VS ? nv - VS : 0; m < nv; ++m)
          mbar_wait(&bars[kVFull + m % VS], (m / VS) & 1, p.err, kDevErrTimeout, nullptr);
        for (int m = nb > BS ? nb - BS : 0; m < nb; ++m)
          mbar_wait(&bars[kBFull + m % BS], (m / BS) & 1, p.err, kDevErrTimeout, nullptr);
      }
    }
  } else if (warp == 1) {
    // ------------------------------------------------------------ MMA issuer
    if (lane == 0 && any_active) {
      bool ok = mbar_wait(&bars[kQFull], 0, p.err, kDevErrTimeout, abort_flag);
      tc_fence_after();
      const uint64_t qdesc = sdesc_sw128(smem_u32(sQ), 16, 1024);
      int n = 0;
      // O += P_m V_m: P from TMEM slot m & 1, V from ring slot m % VS
      auto issue_pv = [&](int m) -> bool {
        const int sm = m & 1, sv = m % VS;
        if (!mbar_wait(&bars[kVFull + sv], (m / VS) & 1, p.err, kDevErrTimeout, abort_flag)) return false;
        if (!mbar_wait(&bars[kPReady + sm], (m >> 1) & 1, p.err, kDevErrTimeout, abort_flag)) return false;
        tc_fence_after();
        const uint64_t vdesc = sdesc_sw128(smem_u32(sV + sv * L::kVB), 16384, 1024);
#pragma unroll
        for (int k = 0; k < 8; ++k)
          umma_ts(tbase + 256, tbase + sm * 128 + k * 8, vdesc + static_cast<uint64_t>((k * 2048) >> 4), IDESC_O,
                  (m > 0 || k > 0) ? 1u : 0u);
        umma_commit(&bars[kVEmpty + sv]);
        umma_commit(&bars[kODone]);
        return true;
      };
      for (int kt = first_kt; ok && kt < p.nTk; kt = next_active(map_row, kt, p.nTk), ++n) {
        const int s = n & 1, sk = n % KS;
        if (!(ok = mbar_wait(&bars[kKFull + sk], (n / KS) & 1, p.err, kDevErrTimeout, abort_flag))) break;
        tc_fence_after();
        const uint64_t kdesc = sdesc_sw128(smem_u32(sK + sk * L::kQB), 16, 1024);
#pragma unroll
        for (int k = 0; k < DQK / 16; ++k)
          umma_ss(tbase + s * 128, qdesc + kmajor_step(k, 128), kdesc + kmajor_step(k, 128), IDESC_S, k > 0);
        umma_commit(&bars[kSFull + s]);
        umma_commit(&bars[kKEmpty + sk]);
        if (n > 0 && !(ok = issue_pv(n - 1))) break;
      }
      if (ok && n > 0) ok = issue_pv(n - 1);
      umma_commit(&bars[kOFinal]);
      umma_commit(&bars[kDrain]);
      mbar_wait(&bars[kDrain], 0, p.err, kDevErrTimeout, nullptr);
    }
  } else {
    // ------------------------------------------------------------ softmax
    const int quad = warp & 3;
    const int r = quad * 32 + lane;
    const int i = q0 + r;
    const uint32_t tl = tbase + (static_cast<uint32_t>(quad * 32) << 16);
    float m_ref = kNegInf, l = 0.f;
    int n = 0;
    // FDMA_FLAG_TEST_SHORT_WAIT: a wait on a barrier nothing arrives at expires first
    bool ok = !p.test_short_wait ||
              mbar_wait(&bars[kFNever], 0, p.err, kDevErrTimeout, abort_flag, kTestWaitNs);
    uint32_t raw[32];
    // Row maximum m_ref in the units of u: u = S*scale + bias with a bias, u = S without one
    // (scale > 0); the softmax exponent in log2 units is u*cexp - m_ref*cexp.
    const float cexp = HAS_BIAS ? kLog2e : p.scale_log2;
    const float thr_u = kRescaleThreshold / cexp;
    const uint64_t c2 = f2(cexp, cexp);
    const uint64_t sc2 = f2(p.scale, p.scale);
    // The keep bits of a partial tile are fetched one active tile ahead, so their load latency
    // overlaps the wait for S.
    auto is_partial = [&](int kt) { return map_row[kt] == kPartial || (ragged_k && kt == p.nTk - 1); };
    uint4 bits_next = make_uint4(~0u, ~0u, ~0u, ~0u);
    if (first_kt < p.nTk && is_partial(first_kt)) bits_next = __ldg(&p.bits_row[(tile_base + first_kt) * kTile + r]);
    for (int kt = first_kt; ok && kt < p.nTk; kt = next_active(map_row, kt, p.nTk), ++n) {
      const int s = n & 1;
      const uint32_t ph = (n >> 1) & 1;
      const bool partial = is_partial(kt);
      const uint4 bits = bits_next;
      {
        const int kn = next_active(map_row, kt, p.nTk);
        bits_next = make_uint4(~0u, ~0u, ~0u, ~0u);
        if (kn < p.nTk && is_partial(kn)) bits_next = __ldg(&p.bits_row[(tile_base + kn) * kTile + r]);
      }
      // Additive term of this tile, formed while S is still being computed: the bias
      // (u = S*scale + bias) and/or -inf at the masked keys (u = S + 0 / -inf).
      const bool addend = HAS_BIAS || partial;
      uint64_t u[64];  // u of keys 2t, 2t+1
      if (HAS_BIAS) {
        const int sb = n % BS;
        if (!(ok = mbar_wait(&bars[kBFull + sb], (n / BS) & 1, p.err, kDevErrTimeout, abort_flag))) break;
        const uint8_t* bt = sB + sb * L::kBB + r * 128;
#pragma unroll
        for (int cc = 0; cc < 16; ++cc) {
          const uint4 bv = *reinterpret_cast<const uint4*>(bt + (cc >> 3) * 16384 + (((cc & 7) ^ (r & 7)) << 4));
          const uint32_t wv[4] = {bv.x, bv.y, bv.z, bv.w};
#pragma unroll
          for (int e = 0; e < 4; ++e) u[cc * 4 + e] = bf16x2_to_f2(wv[e]);
        }
        fence_proxy_async_smem();  // generic reads of the slot before its next TMA write
        mbar_arrive(&bars[kBEmpty + sb]);
      } else if (partial) {
#pragma unroll
        for (int t = 0; t < 64; ++t) u[t] = 0ull;
      }
      if (partial) {
        const uint32_t bw[4] = {bits.x, bits.y, bits.z, bits.w};
#pragma unroll
        for (int t = 0; t < 64; ++t) {
          float u0, u1;
          f2split(u[t], u0, u1);
          if (!((bw[t >> 4] >> ((2 * t) & 31)) & 1u)) u0 = kNegInf;
          if (!((bw[t >> 4] >> ((2 * t + 1) & 31)) & 1u)) u1 = kNegInf;
          u[t] = f2(u0, u1);
        }
      }
      if (!(ok = mbar_wait(&bars[kSFull + s], ph, p.err, kDevErrTimeout, abort_flag))) break;
      tc_fence_after();
#pragma unroll
      for (int c = 0; c < 4; ++c) {
        tmem_ld32(tl + s * 128 + c * 32, raw);
        tmem_ld_wait(raw);
#pragma unroll
        for (int t = 0; t < 16; ++t) {
          const uint64_t s2 = f2(__uint_as_float(raw[2 * t]), __uint_as_float(raw[2 * t + 1]));
          const int q = c * 16 + t;
          u[q] = HAS_BIAS ? fma2(s2, sc2, u[q]) : (addend ? add2(s2, u[q]) : s2);
        }
      }
      float mx8[8];
#pragma unroll
      for (int t = 0; t < 4; ++t) f2split(u[t], mx8[2 * t], mx8[2 * t + 1]);
#pragma unroll
      for (int t = 4; t < 64; t += 4) {
#pragma unroll
        for (int q = 0; q < 4; ++q) {
          float a0, a1;
          f2split(u[t + q], a0, a1);
          // three-input maximum: the running value and both halves of the pair
          asm("max.f32 %0, %0, %1, %2;" : "+f"(mx8[2 * q]) : "f"(a0), "f"(a1));
        }
      }
      float mx;
      asm("max.f32 %0, %1, %2, %3;" : "=f"(mx) : "f"(mx8[0]), "f"(mx8[2]), "f"(mx8[4]));
      asm("max.f32 %0, %0, %1, %2;" : "+f"(mx) : "f"(mx8[6]), "f"(mx8[1]));
      asm("max.f32 %0, %0, %1, %2;" : "+f"(mx) : "f"(mx8[3]), "f"(mx8[5]));
      mx = fmaxf(mx, mx8[7]);
      const float m_new = fmaxf(m_ref, mx);
      float alpha = 1.f;
      bool resc = false;
      if (m_new > m_ref + thr_u) {
        if (m_ref == kNegInf) {
          m_ref = m_new;
        } else {
          alpha = ex2((m_ref - m_new) * cexp);
          l *= alpha;
          m_ref = m_new;
          resc = true;
        }
      }
      if (__any_sync(0xffffffffu, resc)) {
        // O holds P_0..P_{n-1} products: wait for PV_{n-1}, then scale this row.
        if (!(ok = mbar_wait(&bars[kODone], (n - 1) & 1, p.err, kDevErrTimeout, abort_flag))) break;
        tc_fence_after();
#pragma unroll
        for (int c = 0; c < DV / 32; ++c) {
          tmem_ld32(tl + 256 + c * 32, raw);
          tmem_ld_wait(raw);
          uint32_t lo[16], hi[16];
#pragma unroll
          for (int j = 0; j < 16; ++j) {
            lo[j] = __float_as_uint(__uint_as_float(raw[j]) * alpha);
            hi[j] = __float_as_uint(__uint_as_float(raw[16 + j]) * alpha);
          }
          tmem_st16(tl + 256 + c * 32, lo);
          tmem_st16(tl + 256 + c * 32 + 16, hi);
        }
        tmem_st_wait();
      }
      const float nm = (m_ref == kNegInf) ? 0.f : -(m_ref * cexp);
      const uint64_t nm2 = f2(nm, nm);
      float sum4[4] = {0.f, 0.f, 0.f, 0.f};  // (even pairs, odd pairs) x (low, high) halves
#pragma unroll
      for (int c = 0; c < 4; ++c) {
        uint32_t pk[16];
#pragma unroll
        for (int j = 0; j < 16; ++j) {
          float e0, e1;
          f2split(fma2(u[c * 16 + j], c2, nm2), e0, e1);
          const float p0 = ex2(e0), p1 = ex2(e1);
          pk[j] = pack_bf16x2(p0, p1);
          // normalise with the same bf16-rounded weights the PV product uses
          sum4[2 * (j & 1)] = add_bf16lo(pk[j], sum4[2 * (j & 1)]);
          sum4[2 * (j & 1) + 1] = add_bf16hi(pk[j], sum4[2 * (j & 1) + 1]);
        }
        tmem_st16(tl + s * 128 + c * 16, pk);
      }
      l += (sum4[0] + sum4[2]) + (sum4[1] + sum4[3]);
      tmem_st_wait();
      tc_fence_before();
      mbar_arrive(&bars[kPReady + s]);
    }
    // ------------------------------------------------------------ epilogue
    if (ok && n > 0) ok = mbar_wait(&bars[kOFinal], 0, p.err, kDevErrTimeout, abort_flag);
    if (ok) {
      tc_fence_after();
      const float inv = l > 0.f ? 1.f / l : 0.f;
      uint16_t* orow = p.out + ((static_cast<int64_t>(b) * p.Nq + i) * p.Hq + h) * p.dv;
#pragma unroll
      for (int c = 0; c < DV / 32; ++c) {
        if (n > 0) {
          tmem_ld32(tl + 256 + c * 32, raw);
          tmem_ld_wait(raw);
        } else {
#pragma unroll
          for (int j = 0; j < 32; ++j) raw[j] = 0u;
        }
        uint32_t pk[16];
#pragma unroll
        for (int j = 0; j < 16; ++j)
          pk[j] = pack_bf16x2(__uint_as_float(raw[2 * j]) * inv, __uint_as_float(raw[2 * j + 1]) * inv);
        if (i < p.Nq) {  // columns past the head dim are padding
          uint4* dst = reinterpret_cast<uint4*>(orow + c * 32);
#pragma unroll
          for (int v = 0; v < 4; ++v)
            if (c * 32 + v * 8 < p.dv) dst[v] = make_uint4(pk[4 * v], pk[4 * v + 1], pk[4 * v + 2], pk[4 * v + 3]);
        }
      }
      if (i < p.Nq)
        p.lse[(static_cast<int64_t>(b) * p.Hq + h) * p.Nq + i] = l > 0.f ? (m_ref * cexp + log2f(l)) * kLn2 : kNegInf;
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

// ============================================================================
// Two-slot forward (head dims up to 128).  Even GQA group sizes: one CTA = one
// (batch, kv head, 128-row query tile, pair of query heads of the group), and
// both heads read the same K, V, bias and mask tiles, which are fetched once.
// Odd group sizes and MHA (QP): one CTA = one (batch, query head, pair of
// adjacent query tiles 2t, 2t+1); the two tiles share K and V, each has its
// own bias rows and block-map row, and a key tile only one of them needs is
// skipped by the other (the MMA issuer walks the union of the two rows).
// Warps: warpgroup 0 = {TMA producer, MMA issuer, 2 idle}, warpgroup 1 =
// softmax of head 0, warpgroup 2 = softmax of head 1 (setmaxnreg moves
// registers to the softmax groups).  While a softmax warp waits for S it turns
// the tile's bias and keep bits into an additive term (-inf where masked).  The
// MMA issuer interleaves
//   PV0_{n-1} (keys 0..63 as soon as their P is stored, then 64..127), S0_n,
//   PV1_{n-1} (likewise), S1_n
// so each head's softmax overlaps the tensor-core work of the other head, and
// S_w(n) (written over P_w(n-1)'s columns) completes only after PV_w(n-1):
// the softmax may rescale O_w as soon as it sees S_w(n).
// TMEM columns: S0/P0 0..127, S1/P1 128..255, O0 256.., O1 384...
// Shared memory: Q0, Q1; K and V in one 3-slot ring (K_0, V_0, K_1, V_1, ...);
// bias in a 2-slot ring.
enum Fwd2Bar : int {
  k2QFull = 0,
  k2KvFull = 1,    // +slot (3)
  k2KvEmpty = 4,   // +slot (3)
  k2BFull = 7,     // +slot (2)
  k2BEmpty = 9,    // +slot (2)
  k2SFull = 11,    // +head (2)
  k2PReady = 13,   // +2*head+half (4): P of keys 0..63 / 64..127 stored
  k2OFinal = 17,
  k2Drain = 18,
  k2Never = 19,  // never arrived at: the target of the test wait (FDMA_FLAG_TEST_SHORT_WAIT)
  kNumFwd2Bars = 20
};

constexpr int kFwd2Threads = 384;
constexpr uint32_t kFwd2RegsLow = 120, kFwd2RegsHigh = 192;
constexpr int kFwd2MinLaunchRegs = (kFwd2RegsLow + 2 * kFwd2RegsHigh) / 3;  // 168

template <int D, bool HAS_BIAS>
struct Fwd2Smem {
  static constexpr uint32_t kQB = 128u * D * 2u;
  static constexpr uint32_t kBB = 128u * 128u * 2u;
  static constexpr uint32_t kOffQ = 0;                   // [2]
  static constexpr uint32_t kOffKV = 2 * kQB;            // [3]
  static constexpr uint32_t kOffBias = kOffKV + 3 * kQB; // [2]
  static constexpr uint32_t kOffBar = kOffBias + (HAS_BIAS ? 2 * kBB : 0u);
  static constexpr uint32_t kOffMap = kOffBar + kNumFwd2Bars * 8;
  static constexpr uint32_t kOffMisc = kOffMap + kMaxKTiles;
  static constexpr uint32_t kTotal = kOffMisc + 16;
};

// QP (odd group sizes, MHA): the two slots are one head's query tiles 2t and 2t+1 instead of two
// heads of one query tile.  Both slots walk the union of their active key tiles (K and V are the
// same); a tile one slot does not need is fully masked for it (P = 0); each slot has its own
// bias buffer (its own rows), one deep.
template <int D, bool HAS_BIAS, bool QP>
__global__ void __launch_bounds__(kFwd2Threads, 1)
    fwd2_kernel(const __grid_constant__ CUtensorMap tmQ, const __grid_constant__ CUtensorMap tmK,
                const __grid_constant__ CUtensorMap tmV, const __grid_constant__ CUtensorMap tmB,
                const FwdParams p) {
  using L = Fwd2Smem<D, HAS_BIAS>;
  constexpr int KB = D / 64;
  constexpr uint32_t IDESC_S = idesc_bf16(128, 128, false, false);
  constexpr uint32_t IDESC_O = idesc_bf16(128, D, false, true);

  extern __shared__ __align__(1024) uint8_t smem[];
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + L::kOffBar);
  int8_t* map_row = reinterpret_cast<int8_t*>(smem + L::kOffMap);
  uint32_t* misc = reinterpret_cast<uint32_t*>(smem + L::kOffMisc);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(misc + 1);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  int id = blockIdx.x;
  int g, b, h0, qt;
  if (QP) {  // (query-tile pair, head): slot w is query tile 2 * pair + w of head h0
    const int hq = id % p.Hq;
    id /= p.Hq;
    b = id % p.B;
    id /= p.B;
    qt = 2 * (((p.nTq + 1) >> 1) - 1 - id);  // longest causal rows first
    h0 = hq;
    g = hq / p.G;
  } else {  // (query tile, head pair of one group)
    const int GP = p.G >> 1;
    const int hp = id % GP;
    id /= GP;
    g = id % p.Hkv;
    id /= p.Hkv;
    b = id % p.B;
    id /= p.B;
    qt = p.nTq - 1 - id;  // longest causal rows first
    h0 = g * p.G + 2 * hp;
  }
  const int q0 = qt * kTile;
  const int64_t tile_base = (static_cast<int64_t>(b * p.Hkv + g) * p.nTq + qt) * p.nTk;
  const bool ragged_k = (p.Nk & (kTile - 1)) != 0;
  // slot w's query tile (QP: qt + w, possibly past the last tile), head and class of key tile kt
  auto slot_q0 = [&](int w) { return QP ? q0 + w * kTile : q0; };
  auto slot_head = [&](int w) { return QP ? h0 : h0 + w; };
  auto slot_cls = [&](int w, int kt) {
    return QP ? ((map_row[kt] >> (2 * w)) & 3) : static_cast<int>(map_row[kt]);
  };

  if ((smem_u32(smem) & 1023u) != 0) {
    if (threadIdx.x == 0) atomicCAS(p.err, 0, kDevErrAlign);
    return;
  }
  if (threadIdx.x == 0) {
    for (int i = 0; i < kNumFwd2Bars; ++i) mbar_init(&bars[i], 1);
    mbar_init(&bars[k2BEmpty + 0], QP ? 128 : 256);  // QP: each bias buffer serves one slot
    mbar_init(&bars[k2BEmpty + 1], QP ? 128 : 256);
    for (int i = 0; i < 4; ++i) mbar_init(&bars[k2PReady + i], 128);
    misc[1] = 0;
    fence_mbar_init();
  }
  for (int kt = threadIdx.x; kt < p.nTk; kt += blockDim.x) {
    if (QP) {  // both slots' classes: bits 0-1 slot 0, bits 2-3 slot 1 (zero iff both skip)
      const int c0 = p.kmap[tile_base + kt];
      const int c1 = qt + 1 < p.nTq ? p.kmap[tile_base + p.nTk + kt] : kSkip;
      map_row[kt] = static_cast<int8_t>(c0 | (c1 << 2));
    } else {
      map_row[kt] = p.kmap[tile_base + kt];
    }
  }
  if (warp == 1) {
    tmem_alloc(misc, 512);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tbase = misc[0];
  const int first_kt = next_active(map_row, -1, p.nTk);
  const bool any_active = first_kt < p.nTk;

  uint8_t* sQ = smem + L::kOffQ;
  uint8_t* sKV = smem + L::kOffKV;
  uint8_t* sB = smem + L::kOffBias;

  if (warp < 4) {
    regs_decrease<kFwd2RegsLow>();
    if (warp == 0 && lane == 0 && any_active) {
      // ---------------------------------------------------------------- producer
      tma_prefetch_desc(&tmQ);
      tma_prefetch_desc(&tmK);
      tma_prefetch_desc(&tmV);
      if (HAS_BIAS) tma_prefetch_desc(&tmB);
      const uint64_t bias_pol = l2_evict_first();  // each bias tile is read once
      mbar_arrive_expect_tx(&bars[k2QFull], 2 * L::kQB);
#pragma unroll
      for (int w = 0; w < 2; ++w)
#pragma unroll
        for (int c = 0; c < KB; ++c)
          tma_load_4d(sQ + w * L::kQB + c * 16384, &tmQ, &bars[k2QFull], c * 64, slot_q0(w), slot_head(w), b);
      int n = 0, items = 0, nbias = 0;
      int nbw[2] = {0, 0};  // QP: bias fills per slot
      bool ok = true;
      for (int kt = first_kt; ok && kt < p.nTk; kt = next_active(map_row, kt, p.nTk), ++n) {
        const int k0 = kt * kTile;
        // K_n
        {
          const int it = 2 * n, sl = it % 3;
          if (!(ok = mbar_wait(&bars[k2KvEmpty + sl], ((it / 3) & 1) ^ 1, p.err, kDevErrTimeout, abort_flag))) break;
          mbar_arrive_expect_tx(&bars[k2KvFull + sl], L::kQB);
#pragma unroll
          for (int c = 0; c < KB; ++c)
            tma_load_4d(sKV + sl * L::kQB + c * 16384, &tmK, &bars[k2KvFull + sl], c * 64, k0, g, b);
          items = it + 1;
        }
        if (HAS_BIAS && QP) {
          // each slot's own bias rows, into its own buffer (one deep), for the tiles it needs
          for (int w = 0; ok && w < 2; ++w) {
            if (slot_cls(w, kt) == kSkip) continue;
            if (!(ok = mbar_wait(&bars[k2BEmpty + w], (nbw[w] & 1) ^ 1, p.err, kDevErrTimeout, abort_flag))) break;
            mbar_arrive_expect_tx(&bars[k2BFull + w], L::kBB);
#pragma unroll
            for (int c = 0; c < 2; ++c)
              tma_load_4d_hint(sB + w * L::kBB + c * 16384, &tmB, &bars[k2BFull + w], k0 + c * 64, slot_q0(w),
                               g * p.bias_hsel, b * p.bias_bsel, bias_pol);
            ++nbw[w];
          }
          if (!ok) break;
        } else if (HAS_BIAS) {
          const int sb = n & 1;
          if (!(ok = mbar_wait(&bars[k2BEmpty + sb], ((n >> 1) & 1) ^ 1, p.err, kDevErrTimeout, abort_flag))) break;
          mbar_arrive_expect_tx(&bars[k2BFull + sb], L::kBB);
#pragma unroll
          for (int c = 0; c < 2; ++c)
            tma_load_4d_hint(sB + sb * L::kBB + c * 16384, &tmB, &bars[k2BFull + sb], k0 + c * 64, q0, g * p.bias_hsel,
                             b * p.bias_bsel, bias_pol);
          nbias = n + 1;
        }
        // V_n
        {
          const int it = 2 * n + 1, sl = it % 3;
          if (!(ok = mbar_wait(&bars[k2KvEmpty + sl], ((it / 3) & 1) ^ 1, p.err, kDevErrTimeout, abort_flag))) break;
          mbar_arrive_expect_tx(&bars[k2KvFull + sl], L::kQB);
#pragma unroll
          for (int c = 0; c < KB; ++c)
            tma_load_4d(sKV + sl * L::kQB + c * 16384, &tmV, &bars[k2KvFull + sl], c * 64, k0, g, b);
          items = it + 1;
        }
      }
      if (*abort_flag) {
        mbar_wait(&bars[k2QFull], 0, p.err, kDevErrTimeout, nullptr);
        for (int it = items > 3 ? items - 3 : 0; it < items; ++it)
          mbar_wait(&bars[k2KvFull + it % 3], (it / 3) & 1, p.err, kDevErrTimeout, nullptr);
        // and the last fill of each bias slot
        if (QP) {
          for (int w = 0; w < 2; ++w)
            if (nbw[w] > 0) mbar_wait(&bars[k2BFull + w], (nbw[w] - 1) & 1, p.err, kDevErrTimeout, nullptr);
        } else {
          for (int m = nbias > 2 ? nbias - 2 : 0; m < nbias; ++m)
            mbar_wait(&bars[k2BFull + (m & 1)], (m >> 1) & 1, p.err, kDevErrTimeout, nullptr);
        }
      }
    } else if (warp == 1 && lane == 0 && any_active) {
      // ---------------------------------------------------------------- MMA issuer
      bool ok = mbar_wait(&bars[k2QFull], 0, p.err, kDevErrTimeout, abort_flag);
      tc_fence_after();
      const uint64_t qdesc0 = sdesc_sw128(smem_u32(sQ), 16, 1024);
      const uint64_t qdesc1 = sdesc_sw128(smem_u32(sQ + L::kQB), 16, 1024);
      const uint64_t kvk0 = sdesc_sw128(smem_u32(sKV), 16, 1024);       // K-major view of slot 0
      const uint64_t kvmn0 = sdesc_sw128(smem_u32(sKV), 16384, 1024);   // MN-major view of slot 0
      const uint64_t slot_step = static_cast<uint64_t>(L::kQB >> 4);
      auto issue_s = [&](int w, int n) {
        const int sl = (2 * n) % 3;
        const uint64_t kd = kvk0 + sl * slot_step;
        const uint64_t qd = w == 0 ? qdesc0 : qdesc1;
#pragma unroll
        for (int k = 0; k < D / 16; ++k)
          umma_ss(tbase + w * 128, qd + kmajor_step(k, 128), kd + kmajor_step(k, 128), IDESC_S, k > 0);
        umma_commit(&bars[k2SFull + w]);
      };
      // O_w += P_w V, in two key halves, each issued once its P is stored; P of keys
      // 16k .. 16k+15 sits in S_w's columns 8k .. 8k+7
      // (V of union tile m; j = the slot's own P count: its phase and whether O starts here)
      auto pv_when_ready = [&](int w, int m, int j) {
        const int sl = (2 * m + 1) % 3;
        const uint64_t vd = kvmn0 + sl * slot_step;
#pragma unroll
        for (int hf = 0; hf < 2; ++hf) {
          if (!mbar_wait(&bars[k2PReady + 2 * w + hf], j & 1, p.err, kDevErrTimeout, abort_flag)) return false;
          tc_fence_after();
#pragma unroll
          for (int k = hf * 4; k < hf * 4 + 4; ++k)
            umma_ts(tbase + 256 + w * 128, tbase + w * 128 + k * 8, vd + static_cast<uint64_t>((k * 2048) >> 4),
                    IDESC_O, (j > 0 || k > 0) ? 1u : 0u);
        }
        return true;
      };
      int n = 0;
      if constexpr (QP) {
        // Per union tile n: each slot's pending PV (its tile n-1, if it had one) and then, if the
        // slot needs tile n, its S(n).  PV_w always precedes S_w of the slot's next tile.
        int sw[2] = {0, 0};      // S products issued per slot
        bool pend[2] = {false, false};
        for (int kt = first_kt; ok && kt < p.nTk; kt = next_active(map_row, kt, p.nTk), ++n) {
          const int itk = 2 * n;
          for (int w = 0; ok && w < 2; ++w) {
            if (pend[w]) {
              const int itv = 2 * (n - 1) + 1;
              if (!(ok = mbar_wait(&bars[k2KvFull + itv % 3], (itv / 3) & 1, p.err, kDevErrTimeout, abort_flag))) break;
              if (!(ok = pv_when_ready(w, n - 1, sw[w] - 1))) break;
              pend[w] = false;
            }
            if (slot_cls(w, kt) != kSkip) {
              if (!(ok = mbar_wait(&bars[k2KvFull + itk % 3], (itk / 3) & 1, p.err, kDevErrTimeout, abort_flag))) break;
              tc_fence_after();
              issue_s(w, n);
              ++sw[w];
              pend[w] = true;
            }
          }
          if (!ok) break;
          if (n > 0) umma_commit(&bars[k2KvEmpty + (2 * (n - 1) + 1) % 3]);  // V_{n-1}: both slots' PV issued
          umma_commit(&bars[k2KvEmpty + itk % 3]);                            // K_n: read by this tile's S
        }
        if (ok && n > 0) {
          const int itv = 2 * (n - 1) + 1;
          ok = mbar_wait(&bars[k2KvFull + itv % 3], (itv / 3) & 1, p.err, kDevErrTimeout, abort_flag);
          for (int w = 0; ok && w < 2; ++w)
            if (pend[w]) ok = pv_when_ready(w, n - 1, sw[w] - 1);
          if (ok) umma_commit(&bars[k2KvEmpty + itv % 3]);
        }
      }
      for (int kt = first_kt; !QP && ok && kt < p.nTk; kt = next_active(map_row, kt, p.nTk), ++n) {
        const int itk = 2 * n;
        if (n == 0) {
          if (!(ok = mbar_wait(&bars[k2KvFull + itk % 3], (itk / 3) & 1, p.err, kDevErrTimeout, abort_flag))) break;
          tc_fence_after();
          issue_s(0, 0);
          issue_s(1, 0);
          umma_commit(&bars[k2KvEmpty + itk % 3]);
          continue;
        }
        // PV of the previous tile first: it needs only V_{n-1} and P, not K_n (whose
        // ring slot frees only when the tile before that is done)
        const int m = n - 1, itv = 2 * m + 1;
        if (!(ok = mbar_wait(&bars[k2KvFull + itv % 3], (itv / 3) & 1, p.err, kDevErrTimeout, abort_flag))) break;
        if (!(ok = pv_when_ready(0, m, m))) break;
        if (!(ok = mbar_wait(&bars[k2KvFull + itk % 3], (itk / 3) & 1, p.err, kDevErrTimeout, abort_flag))) break;
        tc_fence_after();
        issue_s(0, n);
        if (!(ok = pv_when_ready(1, m, m))) break;
        umma_commit(&bars[k2KvEmpty + itv % 3]);
        issue_s(1, n);
        umma_commit(&bars[k2KvEmpty + itk % 3]);
      }
      if (!QP && ok && n > 0) {
        const int m = n - 1, itv = 2 * m + 1;
        ok = mbar_wait(&bars[k2KvFull + itv % 3], (itv / 3) & 1, p.err, kDevErrTimeout, abort_flag) &&
             pv_when_ready(0, m, m) && pv_when_ready(1, m, m);
        if (ok) umma_commit(&bars[k2KvEmpty + itv % 3]);
      }
      umma_commit(&bars[k2OFinal]);
      umma_commit(&bars[k2Drain]);
      mbar_wait(&bars[k2Drain], 0, p.err, kDevErrTimeout, nullptr);
    }
  } else {
    regs_increase<kFwd2RegsHigh>();
    // ------------------------------------------------------------------ softmax
    const int w = (warp >> 2) - 1;  // slot: head within the pair (QP: query tile within the pair)
    const int h = slot_head(w);
    const int quad = warp & 3;
    const int r = quad * 32 + lane;
    const int i = slot_q0(w) + r;
    const int64_t my_base = tile_base + (QP ? w * p.nTk : 0);  // this slot's row of the block map
    const uint32_t tl = tbase + (static_cast<uint32_t>(quad * 32) << 16);
    const uint32_t scol = w * 128, ocol = 256 + w * 128;
    // Row maximum m_ref is kept in the units of u: u = S*scale + bias with a bias, u = S
    // without one (scale > 0); the softmax exponent in log2 units is u*cexp - m_ref*cexp.
    const float cexp = HAS_BIAS ? kLog2e : p.scale_log2;
    const float thr_u = kRescaleThreshold / cexp;
    const uint64_t c2 = f2(cexp, cexp);
    const uint64_t sc2 = f2(p.scale, p.scale);
    float m_ref = kNegInf, l = 0.f;
    int n = 0;
    // FDMA_FLAG_TEST_SHORT_WAIT: a wait on a barrier nothing arrives at expires first
    bool ok = !p.test_short_wait ||
              mbar_wait(&bars[k2Never], 0, p.err, kDevErrTimeout, abort_flag, kTestWaitNs);
    uint32_t raw[32];
    // The keep bits of a partial tile are fetched one active tile ahead, so their
    // load latency overlaps the wait for S.
    auto is_partial = [&](int kt) {
      if constexpr (QP) {
        const int c = slot_cls(w, kt);
        return c == kPartial || (c == kFull && ragged_k && kt == p.nTk - 1);
      } else {
        return map_row[kt] == kPartial || (ragged_k && kt == p.nTk - 1);
      }
    };
    // this slot's active key tiles (QP: its own row of the block map; otherwise the shared row)
    auto next_mine = [&](int kt) {
      if constexpr (QP) {
        do {
          ++kt;
        } while (kt < p.nTk && slot_cls(w, kt) == kSkip);
        return kt;
      } else {
        return next_active(map_row, kt, p.nTk);
      }
    };
    const int first_mine = QP ? next_mine(-1) : first_kt;
    uint4 bits_next = make_uint4(~0u, ~0u, ~0u, ~0u);
    if (first_mine < p.nTk && is_partial(first_mine)) bits_next = __ldg(&p.bits_row[(my_base + first_mine) * kTile + r]);
    for (int kt = first_mine; ok && kt < p.nTk; kt = next_mine(kt), ++n) {
      const bool partial = is_partial(kt);
      const uint4 bits = bits_next;
      {
        const int kn = next_mine(kt);
        bits_next = make_uint4(~0u, ~0u, ~0u, ~0u);
        if (kn < p.nTk && is_partial(kn)) bits_next = __ldg(&p.bits_row[(my_base + kn) * kTile + r]);
      }
      // Additive term of this tile, formed while S is still being computed: the bias
      // (u = S*scale + bias) and/or -inf at the masked keys (u = S + 0 / -inf).
      // (no bias, QP: the keep bits select on S as it is read, so no u is held across the wait)
      constexpr bool kPreMask = HAS_BIAS || !QP;
      const bool addend = HAS_BIAS || partial;
      uint64_t u[64];  // u of keys 2t, 2t+1
      if (HAS_BIAS) {
        int sb;
        uint32_t bph;
        if constexpr (QP) {  // one fill per own tile, one deep
          sb = w;
          bph = n & 1;
        } else {
          sb = n & 1;
          bph = (n >> 1) & 1;
        }
        if (!(ok = mbar_wait(&bars[k2BFull + sb], bph, p.err, kDevErrTimeout, abort_flag))) break;
        const uint8_t* bt = sB + sb * L::kBB + r * 128;
#pragma unroll
        for (int cc = 0; cc < 16; ++cc) {
          const uint4 bv = *reinterpret_cast<const uint4*>(bt + (cc >> 3) * 16384 + (((cc & 7) ^ (r & 7)) << 4));
          const uint32_t wv[4] = {bv.x, bv.y, bv.z, bv.w};
#pragma unroll
          for (int e = 0; e < 4; ++e) u[cc * 4 + e] = bf16x2_to_f2(wv[e]);
        }
        fence_proxy_async_smem();  // generic reads of the slot before its next TMA write
        mbar_arrive(&bars[k2BEmpty + sb]);
      } else if (kPreMask && partial) {
#pragma unroll
        for (int t = 0; t < 64; ++t) u[t] = 0ull;
      }
      if (kPreMask && partial) {
        const uint32_t bw[4] = {bits.x, bits.y, bits.z, bits.w};
#pragma unroll
        for (int t = 0; t < 64; ++t) {
          float u0, u1;
          f2split(u[t], u0, u1);
          if (!((bw[t >> 4] >> ((2 * t) & 31)) & 1u)) u0 = kNegInf;
          if (!((bw[t >> 4] >> ((2 * t + 1) & 31)) & 1u)) u1 = kNegInf;
          u[t] = f2(u0, u1);
        }
      }
      if (!(ok = mbar_wait(&bars[k2SFull + w], n & 1, p.err, kDevErrTimeout, abort_flag))) break;
      tc_fence_after();
#pragma unroll
      for (int c = 0; c < 4; ++c) {
        tmem_ld32(tl + scol + c * 32, raw);
        tmem_ld_wait(raw);
#pragma unroll
        for (int t = 0; t < 16; ++t) {
          const int q = c * 16 + t;
          if constexpr (kPreMask) {
            const uint64_t s2 = f2(__uint_as_float(raw[2 * t]), __uint_as_float(raw[2 * t + 1]));
            u[q] = HAS_BIAS ? fma2(s2, sc2, u[q]) : (addend ? add2(s2, u[q]) : s2);
          } else {
            float s0 = __uint_as_float(raw[2 * t]), s1 = __uint_as_float(raw[2 * t + 1]);
            if (partial) {
              const uint32_t bw = (q >> 4) == 0 ? bits.x : (q >> 4) == 1 ? bits.y : (q >> 4) == 2 ? bits.z : bits.w;
              if (!((bw >> ((2 * q) & 31)) & 1u)) s0 = kNegInf;
              if (!((bw >> ((2 * q + 1) & 31)) & 1u)) s1 = kNegInf;
            }
            u[q] = f2(s0, s1);
          }
        }
      }
      float mx8[8];
#pragma unroll
      for (int t = 0; t < 4; ++t) f2split(u[t], mx8[2 * t], mx8[2 * t + 1]);
#pragma unroll
      for (int t = 4; t < 64; t += 4) {
#pragma unroll
        for (int q = 0; q < 4; ++q) {
          float a0, a1;
          f2split(u[t + q], a0, a1);
          // three-input maximum: the running value and both halves of the pair
          asm("max.f32 %0, %0, %1, %2;" : "+f"(mx8[2 * q]) : "f"(a0), "f"(a1));
        }
      }
      float mx;
      asm("max.f32 %0, %1, %2, %3;" : "=f"(mx) : "f"(mx8[0]), "f"(mx8[2]), "f"(mx8[4]));
      asm("max.f32 %0, %0, %1, %2;" : "+f"(mx) : "f"(mx8[6]), "f"(mx8[1]));
      asm("max.f32 %0, %0, %1, %2;" : "+f"(mx) : "f"(mx8[3]), "f"(mx8[5]));
      mx = fmaxf(mx, mx8[7]);
      const float m_new = fmaxf(m_ref, mx);
      float alpha = 1.f;
      bool resc = false;
      if (m_new > m_ref + thr_u) {
        if (m_ref == kNegInf) {
          m_ref = m_new;
        } else {
          alpha = ex2((m_ref - m_new) * cexp);
          l *= alpha;
          m_ref = m_new;
          resc = true;
        }
      }
      if (__any_sync(0xffffffffu, resc)) {
        // S_w(n) was issued after PV_w(n-1), so O_w is complete here; PV_w(n) is
        // issued only after the arrivals below, which follow these stores.
#pragma unroll
        for (int c = 0; c < D / 16; ++c) {
          uint32_t o16[16];
          tmem_ld16(tl + ocol + c * 16, o16);
          tmem_ld_wait(o16);
#pragma unroll
          for (int j = 0; j < 16; ++j) o16[j] = __float_as_uint(__uint_as_float(o16[j]) * alpha);
          tmem_st16(tl + ocol + c * 16, o16);
        }
      }
      const float nm = (m_ref == kNegInf) ? 0.f : -(m_ref * cexp);
      const uint64_t nm2 = f2(nm, nm);
      float sum4[4] = {0.f, 0.f, 0.f, 0.f};  // (even pairs, odd pairs) x (low, high) halves
#pragma unroll
      for (int c = 0; c < 4; ++c) {
        uint32_t pk[16];
#pragma unroll
        for (int j = 0; j < 16; ++j) {
          float e0, e1;
          f2split(fma2(u[c * 16 + j], c2, nm2), e0, e1);
          const float p0 = ex2(e0), p1 = ex2(e1);
          pk[j] = pack_bf16x2(p0, p1);
          // the row sum of P as rounded for PV
          sum4[2 * (j & 1)] = add_bf16lo(pk[j], sum4[2 * (j & 1)]);
          sum4[2 * (j & 1) + 1] = add_bf16hi(pk[j], sum4[2 * (j & 1) + 1]);
        }
        tmem_st16(tl + scol + c * 16, pk);
        if (c & 1) {  // keys 0..63 (c = 1), then 64..127 (c = 3): that half of PV may start
          tmem_st_wait();
          tc_fence_before();
          mbar_arrive(&bars[k2PReady + 2 * w + (c >> 1)]);
        }
      }
      {
        l += (sum4[0] + sum4[2]) + (sum4[1] + sum4[3]);
      }
    }
    // ------------------------------------------------------------------ epilogue
    if (ok && n > 0) ok = mbar_wait(&bars[k2OFinal], 0, p.err, kDevErrTimeout, abort_flag);
    if (ok) {
      tc_fence_after();
      const float inv = l > 0.f ? 1.f / l : 0.f;
      uint16_t* orow = p.out + ((static_cast<int64_t>(b) * p.Nq + i) * p.Hq + h) * p.dv;
#pragma unroll
      for (int c = 0; c < D / 32; ++c) {
        if (n > 0) {
          tmem_ld32(tl + ocol + c * 32, raw);
          tmem_ld_wait(raw);
        } else {
#pragma unroll
          for (int j = 0; j < 32; ++j) raw[j] = 0u;
        }
        uint32_t pk[16];
#pragma unroll
        for (int j = 0; j < 16; ++j)
          pk[j] = pack_bf16x2(__uint_as_float(raw[2 * j]) * inv, __uint_as_float(raw[2 * j + 1]) * inv);
        if (i < p.Nq) {  // columns past the head dim are padding
          uint4* dst = reinterpret_cast<uint4*>(orow + c * 32);
#pragma unroll
          for (int v = 0; v < 4; ++v)
            if (c * 32 + v * 8 < p.dv) dst[v] = make_uint4(pk[4 * v], pk[4 * v + 1], pk[4 * v + 2], pk[4 * v + 3]);
        }
      }
      if (i < p.Nq)
        p.lse[(static_cast<int64_t>(b) * p.Hq + h) * p.Nq + i] = l > 0.f ? (m_ref * cexp + log2f(l)) * kLn2 : kNegInf;
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

template <int D, bool HB, bool QP>
cudaError_t launch_fwd2_t(const CUtensorMap& tq, const CUtensorMap& tk, const CUtensorMap& tv, const CUtensorMap& tb,
                          const FwdParams& p, cudaStream_t stream) {
  using L = Fwd2Smem<D, HB>;
  auto kern = fwd2_kernel<D, HB, QP>;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, L::kTotal);
  if (e != cudaSuccess) return e;
  cudaFuncAttributes fa;
  e = cudaFuncGetAttributes(&fa, kern);
  if (e != cudaSuccess) return e;
  if (fa.numRegs < kFwd2MinLaunchRegs) return cudaErrorInvalidConfiguration;  // setmaxnreg split must fit
  const unsigned grid = QP ? static_cast<unsigned>(p.B) * p.Hq * ((p.nTq + 1) / 2)
                           : static_cast<unsigned>(p.B) * p.Hkv * (p.G / 2) * p.nTq;
  kern<<<grid, kFwd2Threads, L::kTotal, stream>>>(tq, tk, tv, tb, p);
  return cudaGetLastError();
}

template <int DQK, int DV, bool HB>
cudaError_t launch_fwd_t(const CUtensorMap& tq, const CUtensorMap& tk, const CUtensorMap& tv, const CUtensorMap& tb,
                         const FwdParams& p, cudaStream_t stream) {
  using L = FwdSmem<DQK, DV, HB>;
  auto kern = fwd_kernel<DQK, DV, HB>;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, L::kTotal);
  if (e != cudaSuccess) return e;
  const unsigned grid = static_cast<unsigned>(p.B) * p.Hq * p.nTq;
  kern<<<grid, 192, L::kTotal, stream>>>(tq, tk, tv, tb, p);
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_fwd(int d, int dv, bool has_bias, const CUtensorMap& tq, const CUtensorMap& tk,
                       const CUtensorMap& tv, const CUtensorMap& tb, const FwdParams& p, cudaStream_t stream) {
  if (d == 192 && dv == 128)
    return has_bias ? launch_fwd_t<192, 128, true>(tq, tk, tv, tb, p, stream)
                    : launch_fwd_t<192, 128, false>(tq, tk, tv, tb, p, stream);
  if (d == 256 && dv == 256)
    return has_bias ? launch_fwd_t<256, 256, true>(tq, tk, tv, tb, p, stream)
                    : launch_fwd_t<256, 256, false>(tq, tk, tv, tb, p, stream);
  if (dv != d) return cudaErrorInvalidValue;
  // even groups: two heads of a group per CTA; odd groups: two query tiles of a head per CTA
  if (p.G % 2 == 0) {
    if (d == 128) return has_bias ? launch_fwd2_t<128, true, false>(tq, tk, tv, tb, p, stream)
                                  : launch_fwd2_t<128, false, false>(tq, tk, tv, tb, p, stream);
    if (d == 64) return has_bias ? launch_fwd2_t<64, true, false>(tq, tk, tv, tb, p, stream)
                                 : launch_fwd2_t<64, false, false>(tq, tk, tv, tb, p, stream);
  }
  if (d == 128) return has_bias ? launch_fwd2_t<128, true, true>(tq, tk, tv, tb, p, stream)
                                : launch_fwd2_t<128, false, true>(tq, tk, tv, tb, p, stream);
  if (d == 64) return has_bias ? launch_fwd2_t<64, true, true>(tq, tk, tv, tb, p, stream)
                               : launch_fwd2_t<64, false, true>(tq, tk, tv, tb, p, stream);
  return cudaErrorInvalidValue;
}

}  // namespace fdma
