// Backward kernels (Flash-DMA issue #73: the backward reuses the forward's
// mask/bias handling and adds the dBias computation; Flash-DMA README, "Key
// Features": forward and backward share the block skip decisions and dBias
// is fused into the backward).
//
//   bwd_pre_kernel   delta_i = <dO_i, O_i> and -lse*log2(e) (-inf for rows with no
//                    kept key and for padding), 32 rows of one head per warp with
//                    coalesced stores; zeroes the fp32 dQ accumulator.
//   bwd_kernel       one CTA = (batch, kv head, 128-key tile).  For every
//                    active query tile (column of the block map, copied into shared
//                    memory) and every query head of the GQA group, one step:
//                      S^T  = K Q^T           (SS, TMEM cols   0..127)
//                      dP^T = V dO^T          (SS, TMEM cols 128..255)
//                      P^T  = exp2(S^T*c + bias^T*log2e - lse2)   (-inf bias at masked
//                                              pairs, or the keep bits without a bias)
//                      scale*dS^T = P^T (scale*dP^T - scale*delta)
//                      dV  += P^T dO          (TS: P^T packed in TMEM cols 0..31, 64..95)
//                      dQ^T = K^T dS^T        (SS: dS^T staged in smem; TMEM cols 128..;
//                                              for d = 64 computed as dQ = dS K)
//                      dK  += dS^T Q          (SS, the same dS^T tile)
//                    Four roles: a TMA producer, a single-thread MMA issuer, two compute
//                    warpgroups and a dQ drain warpgroup.  The compute warps run each step
//                    in two passes, P (right after S^T) and dS (after dP^T); the MMA order
//                    per step is dV(n) once P^T(n) is stored, then S^T(n+1), dQ(n), dK(n),
//                    dP^T(n+1) once dS^T(n) is stored, so the next step's P pass overlaps
//                    the products and the drain reads dQ(n) out of TMEM while dK(n) runs.  The drain warps read dQ out of TMEM and add it to an fp32
//                    accumulator with paced 16-byte reductions.  The softmax scale is folded
//                    into dS (delta comes scaled from the preprocess), so dQ and dK need no
//                    further scaling.  dBias = sum over the group's heads of dS is kept in
//                    registers (one thread per key and half of the query tile) and written
//                    once per (query tile, key tile) through a staged TMA store; the bias
//                    tile of a query tile is TMA-loaded into shared memory once and each
//                    thread copies its key column into registers for all heads.  dO is
//                    double-buffered (with a bias, the second slot is the bias buffer, which a
//                    second producer thread refills with the next tile's bias).  Skipped
//                    tiles of dBias are written as zeros by the same CTA.
//                    Warps: 0 TMA (Q, dO), 1 MMA, 2 TMA (bias), 4..11 two compute groups,
//                    12..15 dQ drain.
//   dq_convert       fp32 accumulator -> bf16 dQ.
#include "fdma_internal.h"
#include "fdma_ptx.cuh"

namespace fdma {
namespace {

constexpr float kLog2e = 1.4426950408889634f;
#define kPosInf (__int_as_float(0x7f800000))

__device__ __forceinline__ float ex2(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

__device__ __forceinline__ float bf16_to_f32(uint32_t h) { return __uint_as_float(h << 16); }

// ----------------------------------------------------------------------- preprocess
// One warp per (batch, head, 32 query rows): delta_i = sum_d dO*O with 16 lanes per row
// (8 bf16 per lane and load), then the 32 rows' -lse*log2(e) and delta are written by one
// coalesced store each.  Each CTA also zeroes a contiguous share of the fp32 dQ accumulator.
constexpr int kPreRowsPerWarp = 32;

__global__ void __launch_bounds__(256) bwd_pre_kernel(const BwdPreParams p) {
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int nblk = (p.nqpad + kPreRowsPerWarp - 1) / kPreRowsPerWarp;
  const int64_t task = static_cast<int64_t>(blockIdx.x) * 8 + warp;  // (b, h, row block), row block fastest
  const int64_t ntask = static_cast<int64_t>(p.B) * p.Hq * nblk;
  if (task < ntask) {
    const int blk = static_cast<int>(task % nblk);
    const int64_t bh = task / nblk;
    const int h = static_cast<int>(bh % p.Hq);
    const int b = static_cast<int>(bh / p.Hq);
    const int i0 = blk * kPreRowsPerWarp;
    const int half = lane >> 4, l16 = lane & 15;
    float mine = 0.f;  // delta of row i0 + lane
#pragma unroll 4
    for (int r = 0; r < kPreRowsPerWarp; r += 2) {
      const int i = i0 + r + half;
      float acc = 0.f;
      if (i < p.Nq) {
        const int64_t off = ((static_cast<int64_t>(b) * p.Nq + i) * p.Hq + h) * p.d;
        for (int c = l16 * 8; c < p.d; c += 128) {
          const uint4 o = *reinterpret_cast<const uint4*>(p.out + off + c);
          const uint4 g = *reinterpret_cast<const uint4*>(p.dout + off + c);
          const uint32_t ow[4] = {o.x, o.y, o.z, o.w}, gw[4] = {g.x, g.y, g.z, g.w};
#pragma unroll
          for (int q = 0; q < 4; ++q)
            acc += bf16_to_f32(ow[q] & 0xFFFFu) * bf16_to_f32(gw[q] & 0xFFFFu) +
                   bf16_to_f32(ow[q] >> 16) * bf16_to_f32(gw[q] >> 16);
        }
      }
#pragma unroll
      for (int o = 8; o > 0; o >>= 1) acc += __shfl_xor_sync(0xffffffffu, acc, o);  // within each half
      const float v0 = __shfl_sync(0xffffffffu, acc, 0), v1 = __shfl_sync(0xffffffffu, acc, 16);
      if (lane == r) mine = v0;
      if (lane == r + 1) mine = v1;
    }
    const int i = i0 + lane;
    if (i < p.nqpad) {
      const int64_t o = (static_cast<int64_t>(b) * p.Hq + h) * p.nqpad + i;
      const bool valid = i < p.Nq;
      float l2 = -kPosInf;
      if (valid) {
        const float l = p.lse[(static_cast<int64_t>(b) * p.Hq + h) * p.Nq + i];
        l2 = (l == -kPosInf) ? -kPosInf : -(l * kLog2e);
      }
      p.lse2[o] = l2;
      p.delta[o] = valid ? -p.scale * mine : 0.f;
    }
  }
  // zero this CTA's contiguous share of the fp32 dQ accumulator
  const int64_t total4 = static_cast<int64_t>(p.B) * p.nqpad * p.Hq * p.dpad / 4;
  const int64_t per = (total4 + gridDim.x - 1) / gridDim.x;
  const int64_t z0 = static_cast<int64_t>(blockIdx.x) * per;
  const int64_t z1 = min(total4, z0 + per);
  float4* z = reinterpret_cast<float4*>(p.dq_acc);
  for (int64_t k = z0 + threadIdx.x; k < z1; k += blockDim.x) z[k] = make_float4(0.f, 0.f, 0.f, 0.f);
}

// Accumulator grouped by four head-dim columns, (B, Hq, dpad/4, nqpad, 4) (64-wide kernels and
// the wide head dims) -> bf16 dQ: one thread per (query, 8 head-dim columns), consecutive
// threads on consecutive queries, so a warp's two 16-byte loads read contiguous bytes; each
// thread stores its 8 columns as 16 bytes.
__global__ void __launch_bounds__(256) dq_convert_grouped_kernel(const DqConvertParams p) {
  const int groups8 = p.dpad >> 3;
  const int64_t idx = static_cast<int64_t>(blockIdx.x) * 256 + threadIdx.x;
  const int64_t total = static_cast<int64_t>(p.B) * p.Hq * groups8 * p.nqpad;
  if (idx >= total) return;
  const int i = static_cast<int>(idx % p.nqpad);
  const int64_t rest = idx / p.nqpad;
  const int c8 = static_cast<int>(rest % groups8);
  const int64_t bh = rest / groups8;
  if (i >= p.Nq || c8 * 8 >= p.d) return;
  const int h = static_cast<int>(bh % p.Hq), b = static_cast<int>(bh / p.Hq);
  const float* src = p.dq_acc + ((bh * (p.dpad >> 2) + 2 * c8) * p.nqpad + i) * 4;
  const float4 a = *reinterpret_cast<const float4*>(src);
  const float4 c = *reinterpret_cast<const float4*>(src + static_cast<int64_t>(p.nqpad) * 4);
  *reinterpret_cast<uint4*>(p.dq + ((static_cast<int64_t>(b) * p.Nq + i) * p.Hq + h) * p.d + c8 * 8) =
      make_uint4(pack_bf16x2(a.x, a.y), pack_bf16x2(a.z, a.w), pack_bf16x2(c.x, c.y), pack_bf16x2(c.z, c.w));
}

// dQ accumulator (interleaved by four queries) -> bf16 dQ for the 128-wide kernels.  A CTA
// converts 32 query rows of one (batch, head): it reads their 16 KB of the accumulator with
// coalesced 16-byte loads into shared memory (4 floats of padding after every 8 head-dim
// indices, so that the transposed reads below hit 32 different banks), then each thread
// packs 8 head-dim indices of one query row and stores them as 16 bytes.
constexpr int kCvtGroups = 8;                 // groups of four query rows per CTA
constexpr int kCvtGroupFloats = 128 * 4 + 64;  // one group in shared memory, padded
__global__ void __launch_bounds__(256) dq_convert4_kernel(const DqConvertParams p) {
  __shared__ __align__(16) float tile[kCvtGroups * kCvtGroupFloats];
  const int nqg = p.nqpad >> 2;
  const int blocks_per_bh = nqg / kCvtGroups;
  const int bh = blockIdx.x / blocks_per_bh;
  const int g0 = (blockIdx.x % blocks_per_bh) * kCvtGroups;
  const int h = bh % p.Hq, b = bh / p.Hq;
  const float4* src = reinterpret_cast<const float4*>(p.dq_acc + (static_cast<int64_t>(bh) * nqg + g0) * 512);
#pragma unroll
  for (int k = 0; k < 4; ++k) {
    const int idx = threadIdx.x + 256 * k;  // group * 128 + head-dim index: its four queries
    const int grp = idx >> 7, c = idx & 127;
    const float4 v = __ldcs(src + idx);     // read once
    *reinterpret_cast<float4*>(&tile[grp * kCvtGroupFloats + c * 4 + (c >> 3) * 4]) = v;
  }
  __syncthreads();
  const int w = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int r4 = lane & 3;
  const int i = (g0 + w) * 4 + r4;  // query row
#pragma unroll
  for (int half = 0; half < 2; ++half) {
    const int c8 = (lane >> 2) + 8 * half;  // head-dim indices 8*c8 .. 8*c8+7
    if (c8 * 8 >= p.d || i >= p.Nq) continue;
    // index 8*c8 + e of query r4 sits at 36*c8 + 4*e + r4 of the group
    const float* t = &tile[w * kCvtGroupFloats + 36 * c8 + r4];
    *reinterpret_cast<uint4*>(p.dq + ((static_cast<int64_t>(b) * p.Nq + i) * p.Hq + h) * p.d + c8 * 8) =
        make_uint4(pack_bf16x2(t[0], t[4]), pack_bf16x2(t[8], t[12]), pack_bf16x2(t[16], t[20]),
                   pack_bf16x2(t[24], t[28]));
  }
}

// ----------------------------------------------------------------------- main backward
enum BwdBar : int {
  kKVFull = 0,
  kQFull = 1,    // +slot (2): Q, lse2, delta of one step
  kQEmpty = 3,   // +slot (2)
  kDoFull = 5,   // +slot (up to 2)
  kDoEmpty = 7,  // +slot (up to 2)
  kBFull = 9,    // bias tile of the current query tile
  kBEmpty = 10,  // the tile's bias has been copied out of the bias buffer (compute threads)
  kSFull = 11,
  kDpFull = 12,
  kPReady = 13,   // P^T of the step stored in TMEM (compute threads)
  kDsReady = 14,  // dS^T of the step stored in shared memory, dP^T read (compute threads)
  kDqFull = 15,
  kDqFree = 16,   // dQ read out of TMEM (drain threads)
  kDsFree = 17,
  kFinal = 18,
  kDrain = 19,
  kNever = 20,    // never arrived at: the target of the test wait (FDMA_FLAG_TEST_SHORT_WAIT)
  kBufDone = 21,  // the last dO of a query tile in the bias buffer has been read (one phase per tile)
  kNumBwdBars = 22
};

// 16 warps: warpgroup 0 = {TMA producer, MMA issuer, 2 idle}, warpgroups 1-2 = compute,
// warpgroup 3 = dQ drain.  setmaxnreg moves registers from warpgroup 0 to the others; the
// four shares add up to the 128 registers per thread the kernel is launched with.
constexpr int kBwdThreads = 512;
constexpr unsigned kDrainPaceNs = 32;  // pause after each 16-byte dQ reduction of a drain thread
constexpr uint32_t kRegsCtl = 48, kRegsCompute = 160, kRegsDrain = 144;
// With a bias at d = 128 the compute warps also hold the tile's bias column: 8 more registers
// there (taken from the control warpgroup) leave fewer spills and a 1.6 % faster backward at
// N=16384; without a bias the same split made the document-mask backward 1.2 % slower.
constexpr uint32_t kRegsCtlB = 32, kRegsComputeB = 168;
constexpr int kBwdMinLaunchRegs = (kRegsCtl + 2 * kRegsCompute + kRegsDrain) / 4;  // 128
static_assert(kBwdMinLaunchRegs * kBwdThreads <= 65536, "register split exceeds the register file");
static_assert(kRegsCtlB + 2 * kRegsComputeB == kRegsCtl + 2 * kRegsCompute, "both splits fill the same launch");

// Shared memory: K, V resident; Q (+ lse, delta) in 2 slots; dO in 1 slot when a
// bias tile needs the room, else 2; bias tile (one query tile, 32 KB); dS^T.
template <int D, bool HAS_BIAS>
struct BwdSmem {
  static constexpr uint32_t kQB = 128u * D * 2u;
  static constexpr int kDoStages = HAS_BIAS ? 1 : 2;
  static constexpr uint32_t kOffK = 0;
  static constexpr uint32_t kOffV = kQB;
  static constexpr uint32_t kOffQ = 2 * kQB;                      // [2]
  static constexpr uint32_t kOffDO = 4 * kQB;                     // [kDoStages]
  static constexpr uint32_t kOffBias = kOffDO + kDoStages * kQB;  // 128 x 128 bf16 (if HAS_BIAS)
  static constexpr uint32_t kOffDS = kOffBias + (HAS_BIAS ? 32768u : 0u);  // 128 keys x 128 queries bf16
  static constexpr uint32_t kOffLse = kOffDS + 32768;    // [2][128] f32
  static constexpr uint32_t kOffDelta = kOffLse + 1024;  // [2][128] f32
  static constexpr uint32_t kOffBar = kOffDelta + 1024;
  static constexpr uint32_t kOffMisc = kOffBar + kNumBwdBars * 8;
  static constexpr uint32_t kOffMap = kOffMisc + 16;  // this key tile's column of the block map, 2 bits per query tile
  static constexpr uint32_t kTotal = kOffMap + kMaxKTiles / 4;
  static_assert(kTotal <= 232448, "bwd shared memory exceeds the per-CTA limit");
};

// Descriptor offsets (16-byte units) of the k-th 16-element K step of a 128-row SW128 tile
// made of 64-column blocks: K-major (K along the 128-byte rows) and MN-major (K across rows).
__host__ __device__ constexpr uint32_t kmajor_off(int k) {
  return static_cast<uint32_t>(((k >> 2) * 128u * 128u + (k & 3) * 32u) >> 4);
}
__host__ __device__ constexpr uint32_t mnmajor_off(int k) { return static_cast<uint32_t>((k * 2048) >> 4); }

// The active query tiles of one key-tile column of the block map, from a shared-memory
// copy packed 2 bits per query tile (kSkip / kPartial / kFull), in increasing order.
struct ColIter {
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

// dO slot of step n (head hh of its query tile).  Without a bias there are two dO slots,
// used alternately.  With a bias the second slot is the bias buffer (it directly follows the
// dO slot), which holds a query tile's bias until the compute warps have copied it (right
// before the tile's first step): the first and the last head of every tile use slot 0, the
// heads between alternate, so the buffer's last dO use in a tile comes early and the next
// tile's bias has time to arrive.  With G = 4: slots 0, 1, 0, 0.
template <bool HAS_BIAS>
__device__ __forceinline__ int do_slot(int n, int hh, int G) {
  return HAS_BIAS ? ((hh == G - 1) ? 0 : (hh & 1)) : (n & 1);
}
// Number of slot-1 (bias buffer) dO fills in one query tile under do_slot with a bias, and the
// head of the last of them (-1 when there is none).
__device__ __forceinline__ int slot1_fills_per_tile(int G) { return (G - 1) / 2; }
__device__ __forceinline__ int last_slot1_head(int G) { return G >= 3 ? (((G - 2) & 1) ? G - 2 : G - 3) : -1; }

template <int D, bool HAS_BIAS, bool WANT_DBIAS>
__global__ void __launch_bounds__(kBwdThreads, 1)
    bwd_kernel(const __grid_constant__ CUtensorMap tmQ, const __grid_constant__ CUtensorMap tmK,
               const __grid_constant__ CUtensorMap tmV, const __grid_constant__ CUtensorMap tmDO,
               const __grid_constant__ CUtensorMap tmB, const __grid_constant__ CUtensorMap tmDB,
               const BwdParams p) {
  using L = BwdSmem<D, HAS_BIAS>;
  constexpr int KB = D / 64;
  constexpr bool DQ_T = (D == 128);  // dQ^T = K^T dS^T (lane = head-dim index) for coalesced reductions
  constexpr uint32_t IDESC_S = idesc_bf16(128, 128, false, false);   // S^T, dP^T
  constexpr uint32_t IDESC_DV = idesc_bf16(128, D, false, true);     // P^T(tmem) x dO (N contiguous)
  constexpr uint32_t IDESC_DK = idesc_bf16(128, D, false, true);     // dS^T (K contiguous) x Q (N contiguous)
  constexpr uint32_t IDESC_DQ = DQ_T ? idesc_bf16(128, 128, true, true)   // K^T (M=d contiguous) x dS^T
                                     : idesc_bf16(128, D, true, true);    // dS (M contiguous) x K

  extern __shared__ __align__(1024) uint8_t smem[];
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + L::kOffBar);
  uint32_t* misc = reinterpret_cast<uint32_t*>(smem + L::kOffMisc);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(misc + 1);
  uint8_t* sK = smem + L::kOffK;
  uint8_t* sV = smem + L::kOffV;
  uint8_t* sQ = smem + L::kOffQ;
  uint8_t* sDO = smem + L::kOffDO;
  uint8_t* sBias = smem + L::kOffBias;
  uint8_t* sDS = smem + L::kOffDS;
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
  const ColIter it{map2, p.nTq};
  const bool ragged_k = (p.Nk & (kTile - 1)) != 0 && kt == p.nTk - 1;
  const bool ragged_q_any = (p.Nq & (kTile - 1)) != 0;

  if ((smem_u32(smem) & 1023u) != 0) {
    if (threadIdx.x == 0) atomicCAS(p.err, 0, kDevErrAlign);
    return;
  }
  if (threadIdx.x == 0) {
    for (int i = 0; i < kNumBwdBars; ++i) mbar_init(&bars[i], 1);
    mbar_init(&bars[kBEmpty], 256);
    mbar_init(&bars[kPReady], 256);
    mbar_init(&bars[kDsReady], 256);
    mbar_init(&bars[kDqFree], 128);
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
   regs_decrease<(D == 128 && HAS_BIAS) ? kRegsCtlB : kRegsCtl>();
   if (warp == 0 && lane == 0 && any_active) {
    // ------------------------------------------------------------ producer
    tma_prefetch_desc(&tmQ);
    tma_prefetch_desc(&tmK);
    tma_prefetch_desc(&tmV);
    tma_prefetch_desc(&tmDO);
    mbar_arrive_expect_tx(&bars[kKVFull], 2 * L::kQB);
#pragma unroll
    for (int c = 0; c < KB; ++c) {
      tma_load_4d(sK + c * 16384, &tmK, &bars[kKVFull], c * 64, k0, g, b);
      tma_load_4d(sV + c * 16384, &tmV, &bars[kKVFull], c * 64, k0, g, b);
    }
    int n = 0, qi_count = 0, nq_issued = 0;
    int ufill0 = 0, ufill1 = 0;  // dO fills of slot 0 / slot 1
    bool ok = true;
    for (int qt = first_qt; ok && it.valid(qt); qt = it.next(qt), ++qi_count) {
      for (int hh = 0; hh < p.G; ++hh, ++n) {
        const int h = g * p.G + hh;
        const int s = n & 1;
        if (!(ok = mbar_wait(&bars[kQEmpty + s], ((n >> 1) & 1) ^ 1, p.err, kDevErrTimeout, abort_flag))) break;
        mbar_arrive_expect_tx(&bars[kQFull + s], L::kQB + 1024);
#pragma unroll
        for (int c = 0; c < KB; ++c)
          tma_load_4d(sQ + s * L::kQB + c * 16384, &tmQ, &bars[kQFull + s], c * 64, qt * kTile, h, b);
        const int64_t vec = (static_cast<int64_t>(b) * p.Hq + h) * p.nqpad + qt * kTile;
        bulk_load(sLse + s * 128, p.lse2 + vec, 512, &bars[kQFull + s]);
        bulk_load(sDelta + s * 128, p.delta + vec, 512, &bars[kQFull + s]);
        nq_issued = n + 1;
        const int sd = do_slot<HAS_BIAS>(n, hh, p.G);
        const int u = sd ? ufill1 : ufill0;
        if (HAS_BIAS && sd == 1 && hh == 1) {
          // first dO in the bias buffer this tile: the tile's bias must have been copied out
          if (!(ok = mbar_wait(&bars[kBEmpty], qi_count & 1, p.err, kDevErrTimeout, abort_flag))) break;
        } else {
          if (!(ok = mbar_wait(&bars[kDoEmpty + sd], (u & 1) ^ 1, p.err, kDevErrTimeout, abort_flag))) break;
        }
        mbar_arrive_expect_tx(&bars[kDoFull + sd], L::kQB);
#pragma unroll
        for (int c = 0; c < KB; ++c)
          tma_load_4d(sDO + sd * L::kQB + c * 16384, &tmDO, &bars[kDoFull + sd], c * 64, qt * kTile, h, b);
        if (sd) ufill1 = u + 1;
        else ufill0 = u + 1;
      }
      if (!ok) break;
    }
    if (*abort_flag) {
      // let this CTA's own copies land before it retires (bounded waits)
      mbar_wait(&bars[kKVFull], 0, p.err, kDevErrTimeout, nullptr);
      for (int m = nq_issued > 2 ? nq_issued - 2 : 0; m < nq_issued; ++m)
        mbar_wait(&bars[kQFull + (m & 1)], (m >> 1) & 1, p.err, kDevErrTimeout, nullptr);
      // only the last fill of each slot can still be in flight
      if (ufill0 > 0) mbar_wait(&bars[kDoFull + 0], (ufill0 - 1) & 1, p.err, kDevErrTimeout, nullptr);
      if (ufill1 > 0) mbar_wait(&bars[kDoFull + 1], (ufill1 - 1) & 1, p.err, kDevErrTimeout, nullptr);
    }
   } else if (HAS_BIAS && warp == 2 && lane == 0 && any_active) {
    // ------------------------------------------------------------ bias producer
    // One bias tile per active query tile into the bias buffer: the first at once, each
    // later one as soon as the buffer is free, i.e. once the last dO that went into the
    // buffer during the previous tile has been read by its products (or, with no such dO,
    // once the previous tile's bias has been copied out).
    tma_prefetch_desc(&tmB);
    const uint64_t bias_pol = l2_evict_first();  // each bias tile is read once here
    const int per_tile = slot1_fills_per_tile(p.G);
    int nbias = 0;
    bool ok = true;
    for (int qt = first_qt; ok && it.valid(qt); qt = it.next(qt)) {
      if (nbias > 0) {
        // kBufDone completes once per tile (an mbarrier parity wait must not fall two phases
        // behind, so the per-fill kDoEmpty phases are not waited on here)
        if (per_tile > 0)
          ok = mbar_wait(&bars[kBufDone], (nbias - 1) & 1, p.err, kDevErrTimeout, abort_flag);
        else
          ok = mbar_wait(&bars[kBEmpty], (nbias - 1) & 1, p.err, kDevErrTimeout, abort_flag);
        if (!ok) break;
      }
      mbar_arrive_expect_tx(&bars[kBFull], 32768);
#pragma unroll
      for (int c = 0; c < 2; ++c)
        tma_load_4d_hint(sBias + c * 16384, &tmB, &bars[kBFull], k0 + c * 64, qt * kTile, g * p.bias_hsel,
                         b * p.bias_bsel, bias_pol);
      ++nbias;
    }
    // only the last bias fill can still be in flight
    if (*abort_flag && nbias > 0) mbar_wait(&bars[kBFull], (nbias - 1) & 1, p.err, kDevErrTimeout, nullptr);
   } else if (warp == 1 && lane == 0 && any_active) {
    // ------------------------------------------------------------ MMA issuer
    bool ok = mbar_wait(&bars[kKVFull], 0, p.err, kDevErrTimeout, abort_flag);
    tc_fence_after();
    const uint64_t kdesc_k = sdesc_sw128(smem_u32(sK), 16, 1024);
    const uint64_t vdesc_k = sdesc_sw128(smem_u32(sV), 16, 1024);
    const uint64_t kdesc_mn = sdesc_sw128(smem_u32(sK), 16384, 1024);
    const uint64_t dsdesc_mn = sdesc_sw128(smem_u32(sDS), 16384, 1024);
    const uint64_t dsdesc_k = sdesc_sw128(smem_u32(sDS), 16, 1024);
    const uint64_t q0desc_k = sdesc_sw128(smem_u32(sQ), 16, 1024);
    const uint64_t q0desc_mn = sdesc_sw128(smem_u32(sQ), 16384, 1024);
    const uint64_t do0desc_k = sdesc_sw128(smem_u32(sDO), 16, 1024);
    const uint64_t do0desc_mn = sdesc_sw128(smem_u32(sDO), 16384, 1024);
    const uint64_t slot = static_cast<uint64_t>(L::kQB >> 4);
    int n = 0;
    int uuse0 = 0, uuse1 = 0;  // dO uses of slot 0 / slot 1
    // S^T of step m (query slot m & 1) into columns 0..127; false after a failed wait
    auto issue_s = [&](int m) -> bool {
      const int s = m & 1;
      if (!mbar_wait(&bars[kQFull + s], (m >> 1) & 1, p.err, kDevErrTimeout, abort_flag)) return false;
      tc_fence_after();
      const uint64_t qdesc_k = q0desc_k + s * slot;
      static_for<0, D / 16>([&](auto kc) {
        constexpr int k = decltype(kc)::value;
        umma_ss_off<kmajor_off(k), kmajor_off(k)>(tbase, kdesc_k, qdesc_k, IDESC_S, k > 0);
      });
      umma_commit(&bars[kSFull]);
      return true;
    };
    // dP^T of step m (dO slot sd) into columns 128..255, which the previous dQ used
    auto issue_dp = [&](int m, int sd) -> bool {
      const uint64_t dodesc_k = do0desc_k + sd * slot;
      if (!mbar_wait(&bars[kDoFull + sd], (sd ? uuse1 : uuse0) & 1, p.err, kDevErrTimeout, abort_flag)) return false;
      if (m > 0 && !mbar_wait(&bars[kDqFree], (m - 1) & 1, p.err, kDevErrTimeout, abort_flag)) return false;
      tc_fence_after();
      static_for<0, D / 16>([&](auto kc) {
        constexpr int k = decltype(kc)::value;
        umma_ss_off<kmajor_off(k), kmajor_off(k)>(tbase + 128, vdesc_k, dodesc_k, IDESC_S, k > 0);
      });
      umma_commit(&bars[kDpFull]);
      return true;
    };
    // Per step n: dV(n) as soon as P^T(n) is stored (it overlaps the dS pass), then, once
    // dS^T(n) is stored, S^T(n+1), dQ(n), dK(n), dP^T(n+1).  The compute warps start on
    // P^T(n+1) as soon as S^T(n+1) is done; the drain warps read dQ(n) out of TMEM (over the
    // dP^T columns) while dK(n) runs, so dP^T(n+1) can follow dK(n) at once.  dQ(n) and dK(n)
    // both take dS^T from shared memory; dK(n) frees the Q slot for the load two steps ahead.
    ok = ok && issue_s(0) && issue_dp(0, do_slot<HAS_BIAS>(0, 0, p.G));
    for (int qt = first_qt; ok && it.valid(qt); qt = it.next(qt)) {
      for (int hh = 0; hh < p.G; ++hh, ++n) {
        const int s = n & 1, sd = do_slot<HAS_BIAS>(n, hh, p.G);
        const uint64_t qdesc_mn = q0desc_mn + s * slot, dodesc_mn = do0desc_mn + sd * slot;
        if (!(ok = mbar_wait(&bars[kPReady], n & 1, p.err, kDevErrTimeout, abort_flag))) break;
        tc_fence_after();
        // dV += P^T dO  (K dimension = 128 queries; P^T packed in TMEM cols 0..31 and 64..95)
        static_for<0, 8>([&](auto kc) {
          constexpr int k = decltype(kc)::value;
          umma_ts_off<k * 8 + (k >= 4 ? 32 : 0), mnmajor_off(k)>(tbase + 256, tbase, dodesc_mn, IDESC_DV,
                                                                  (n > 0 || k > 0) ? 1u : 0u);
        });
        umma_commit(&bars[kDoEmpty + sd]);  // dP^T(n) and dV(n) have read this dO slot
        if (HAS_BIAS && hh == last_slot1_head(p.G)) umma_commit(&bars[kBufDone]);  // the buffer's last dO this tile
        if (sd) ++uuse1;
        else ++uuse0;
        if (!(ok = mbar_wait(&bars[kDsReady], n & 1, p.err, kDevErrTimeout, abort_flag))) break;
        tc_fence_after();
        const bool more = hh + 1 < p.G || it.valid(it.next(qt));
        if (more && !(ok = issue_s(n + 1))) break;  // over P^T(n), which dV(n) and the dS pass have read
        // dQ (K dimension = 128 keys) over the dP^T columns, first: the drain reads it out of
        // TMEM while dK runs
        static_for<0, 8>([&](auto kc) {
          constexpr int k = decltype(kc)::value;
          if (DQ_T)
            umma_ss_off<mnmajor_off(k), mnmajor_off(k)>(tbase + 128, kdesc_mn, dsdesc_mn, IDESC_DQ, k > 0);
          else
            umma_ss_off<mnmajor_off(k), mnmajor_off(k)>(tbase + 128, dsdesc_mn, kdesc_mn, IDESC_DQ, k > 0);
        });
        umma_commit(&bars[kDqFull]);
        // dK += dS^T Q  (SS: dS^T K-major in shared memory)
        static_for<0, 8>([&](auto kc) {
          constexpr int k = decltype(kc)::value;
          umma_ss_off<kmajor_off(k), mnmajor_off(k)>(tbase + 384, dsdesc_k, qdesc_mn, IDESC_DK, (n > 0 || k > 0) ? 1u : 0u);
        });
        umma_commit(&bars[kQEmpty + s]);
        umma_commit(&bars[kDsFree]);  // the shared-memory dS^T tile has been read
        if (more) {
          const int hn = hh + 1 < p.G ? hh + 1 : 0;
          if (!(ok = issue_dp(n + 1, do_slot<HAS_BIAS>(n + 1, hn, p.G)))) break;
        }
      }
    }
    umma_commit(&bars[kFinal]);
    umma_commit(&bars[kDrain]);
    mbar_wait(&bars[kDrain], 0, p.err, kDevErrTimeout, nullptr);
   }
  } else if (warp < 12) {
   regs_increase<(D == 128 && HAS_BIAS) ? kRegsComputeB : kRegsCompute>();
   {
    // ------------------------------------------------------------ compute
    // Two warpgroups: wg 0 owns queries 0..63 of every step, wg 1 queries 64..127.
    // Thread (quad, lane) owns key row j of S^T/dP^T/dK/dV.  Per step: the P pass (S^T ->
    // P^T, packed bf16 into this warpgroup's own S^T columns), then the dS pass (P^T and
    // dP^T -> scale * dS^T into shared memory, dBias partial sums in registers).
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
    const uint64_t lg2 = f2(kLog2e, kLog2e);
    int n = 0, qi_count = 0;
    // With FDMA_FLAG_TEST_SHORT_WAIT every compute thread first waits on a barrier that
    // nothing arrives at, with a short limit: the wait expires, records FDMA_ERR_TIMEOUT and
    // raises the abort flag, and the CTA unwinds as after any expired wait.
    bool ok = !p.test_short_wait ||
              mbar_wait(&bars[kNever], 0, p.err, kDevErrTimeout, abort_flag, kTestWaitNs);
    // No compute thread leaves these loops early, so every one of them reaches every named
    // barrier below; after a failed wait (ok == false) the work and the stores are skipped.
    // Per query tile: the keep bits of queries qbase..qbase+63 for key j and the bias^T column
    // slice, copied once into registers for every head (only the P passes use them).
    uint32_t bw0 = ~0u, bw1 = ~0u;
    uint32_t bpk[HAS_BIAS ? 32 : 1];
    // keep bits of queries qbase..qbase+63 for key j in query tile qt (all ones unless partial)
    auto load_bits = [&](int qt) -> uint2 {
      uint2 bb = make_uint2(~0u, ~0u);
      if (it.valid(qt) && (it.cls(qt) == kPartial || ragged_k || (ragged_q_any && qt == p.nTq - 1))) {
        const int64_t tile = col_base + static_cast<int64_t>(qt) * p.nTk;
        bb = reinterpret_cast<const uint2*>(&p.bits_col[tile * kTile + j])[wg];
      }
      return bb;
    };
    // the tile's keep bits (loaded one tile ahead) and bias^T slice, into registers
    auto fetch_tile = [&](const uint2 bits, int qi) {
      bw0 = bits.x;
      bw1 = bits.y;
      if (HAS_BIAS) {
        ok = ok && mbar_wait(&bars[kBFull], qi & 1, p.err, kDevErrTimeout, abort_flag);
        const uint8_t* bt = sBias + (j >> 6) * 16384 + (j & 7) * 2;
        const int jc = (j & 63) >> 3;
#pragma unroll
        for (int e = 0; e < 32; ++e) {
          const int i0 = qbase + 2 * e, i1 = i0 + 1;
          const uint32_t lo = *reinterpret_cast<const uint16_t*>(bt + i0 * 128 + ((jc ^ (i0 & 7)) << 4));
          const uint32_t hi = *reinterpret_cast<const uint16_t*>(bt + i1 * 128 + ((jc ^ (i1 & 7)) << 4));
          // masked (query, key) pairs get a bias of -inf (bf16 0xFF80): their P is exp2(-inf) = 0
          const uint32_t wd = e < 16 ? bw0 : bw1;
          const bool k0b = (wd >> ((2 * e) & 31)) & 1u, k1b = (wd >> ((2 * e + 1) & 31)) & 1u;
          bpk[e] = (k0b ? lo : 0xFF80u) | ((k1b ? hi : 0xFF80u) << 16);
        }
        // The buffer is next written by TMA (the async proxy): the proxy fence orders these
        // generic reads before that write.  Without it the write was seen to overtake reads
        // still in flight (head dim 64, dO into the buffer right after the release).
        fence_proxy_async_smem();
        mbar_arrive(&bars[kBEmpty]);
      }
    };
    // Write the summed dBias of the query tile at q0t straight from registers, pairs of
    // queries qp0 .. qp0+NP-1: thread (key j) holds its key's column slice (64 queries); one
    // lane shuffle per pair of queries trades halves with the neighbouring key so that each
    // thread stores two adjacent keys of one row (4 bytes), and a warp instruction writes two
    // contiguous 64-byte row segments.
    auto store_dbias = [&](int q0t, int qp0, auto npc) {
      constexpr int NP = decltype(npc)::value;
      const uint64_t inv2 = f2(1.f / p.scale, 1.f / p.scale);  // the sums are of scale * dS
      const bool odd = (j & 1) != 0;
      const int col = kidx & ~1;  // this thread's pair of keys: col, col + 1
      uint32_t* base = reinterpret_cast<uint32_t*>(
          p.dbias + ((static_cast<int64_t>(b) * p.Hkv + g) * p.Nq + q0t + qbase + (odd ? 1 : 0)) * p.Nk + col);
      const int64_t row2 = p.Nk;  // two rows of bf16, in 4-byte words
#pragma unroll
      for (int qp = qp0; qp < qp0 + NP; ++qp) {
        float a0, a1;
        f2split(mul2(acc2[qp], inv2), a0, a1);
        const uint32_t w = pack_bf16x2(a0, a1);  // (query 2qp, query 2qp+1) of key j
        // even key: keeps its row-2qp value, sends its row-2qp+1 value; odd key the reverse
        const uint32_t send = odd ? (w & 0xFFFFu) : (w >> 16);
        const uint32_t got = __shfl_xor_sync(0xffffffffu, send, 1);
        // row 2qp (even thread): (key col, key col+1) = (w.lo, got); row 2qp+1 (odd thread):
        // (key col, key col+1) = (got, w.hi)
        const uint32_t pair = odd ? (got | (w & 0xFFFF0000u)) : ((w & 0xFFFFu) | (got << 16));
        const int row = q0t + qbase + 2 * qp + (odd ? 1 : 0);
        if (ok && row < p.Nq && kin) base[qp * row2] = pair;
        acc2[qp] = 0ull;
      }
    };
    int q0_prev = 0;
    uint2 bits_next = load_bits(first_qt);
    for (int qt = first_qt; it.valid(qt); qt = it.next(qt), ++qi_count) {
      const int q0 = qt * kTile;
      // the previous tile's dBias (complete after its last dS pass), then this tile's keep
      // bits and bias^T slice, right before its first P pass; the next tile's keep bits are
      // requested now so that their load is hidden behind this tile's steps
      if (WANT_DBIAS && qi_count > 0) store_dbias(q0_prev, 0, std::integral_constant<int, 32>{});
      fetch_tile(bits_next, qi_count);
      bits_next = load_bits(it.next(qt));
      for (int hh = 0; hh < p.G; ++hh, ++n) {
        const int s = n & 1;
        // ---------------- P pass: P^T = exp2(S^T * scale*log2e + bias^T*log2e - lse*log2e)
        ok = ok && mbar_wait(&bars[kSFull], n & 1, p.err, kDevErrTimeout, abort_flag);
        ok = ok && mbar_wait(&bars[kQFull + s], (n >> 1) & 1, p.err, kDevErrTimeout, abort_flag);
        if (ok) {
          tc_fence_after();
          const float* lse2 = sLse + s * 128 + qbase;
#pragma unroll
          for (int c = 0; c < 4; ++c) {  // 16 queries per chunk
            const int col = qbase + c * 16;
            uint32_t sr[16];
            tmem_ld16(tl + col, sr);
            uint64_t nl[8];  // this chunk's 16 -lse*log2(e) values as pairs (broadcast 16-byte reads)
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
              const int qi = c * 16 + e;  // 0..63 within this half (even)
              const uint64_t s2 = f2(__uint_as_float(sr[e]), __uint_as_float(sr[e + 1]));
              const uint64_t x2 = HAS_BIAS ? fma2(s2, sc2, fma2(bf16x2_to_f2(bpk[qi >> 1]), lg2, nl[e >> 1]))
                                           : fma2(s2, sc2, nl[e >> 1]);
              float x0, x1;
              f2split(x2, x0, x1);
              // with a bias the keep bits are already folded into it as -inf
              const float p0 = (HAS_BIAS || ((word >> (qi & 31)) & 1u)) ? ex2(x0) : 0.f;
              const float p1 = (HAS_BIAS || ((word >> ((qi + 1) & 31)) & 1u)) ? ex2(x1) : 0.f;
              pk[e >> 1] = pack_bf16x2(p0, p1);
            }
            // packed P^T stays inside this warpgroup's own S^T columns (already read):
            // queries 0..63 -> cols 0..31, queries 64..127 -> cols 64..95
            tmem_st8(tl + wg * 64 + c * 8, pk);
          }
          tmem_st_wait();
          tc_fence_before();
          mbar_arrive(&bars[kPReady]);
        }
        // ---------------- dS pass: scale * dS^T = P^T (scale * dP^T - scale * delta)
        ok = ok && mbar_wait(&bars[kDpFull], n & 1, p.err, kDevErrTimeout, abort_flag);
        if (ok) {
          tc_fence_after();
          const float* dlt = sDelta + s * 128 + qbase;
#pragma unroll
          for (int c = 0; c < 4; ++c) {
            const int col = qbase + c * 16;
            uint32_t pp[8], dr[16];
            tmem_ld8(tl + wg * 64 + c * 8, pp);
            tmem_ld16(tl + 128 + col, dr);
            uint64_t dd[8];  // this chunk's 16 -scale*delta values as pairs
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
              const int qi = c * 16 + e;
              // scale * dS = P * (scale * dP - scale * delta): the scale of dQ and dK is applied here
              const uint64_t dv2 = mul2(bf16x2_to_f2(pp[e >> 1]),
                                        fma2(f2(__uint_as_float(dr[e]), __uint_as_float(dr[e + 1])), scl2, dd[e >> 1]));
              if (WANT_DBIAS) acc2[qi >> 1] = add2(acc2[qi >> 1], dv2);
              float d0, d1;
              f2split(dv2, d0, d1);
              dk[e >> 1] = pack_bf16x2(d0, d1);
            }
            // the previous step's dQ and dK must have read the shared-memory dS^T tile
            if (c == 0 && n > 0 && !mbar_wait(&bars[kDsFree], (n - 1) & 1, p.err, kDevErrTimeout, abort_flag)) {
              ok = false;
              break;
            }
            // dS^T row j, queries col..col+15: two 16-byte chunks of the SW128 K-major tile
            uint8_t* rowp = sDS + wg * 16384 + j * 128;
            *reinterpret_cast<uint4*>(rowp + (((2 * c) ^ (j & 7)) << 4)) = make_uint4(dk[0], dk[1], dk[2], dk[3]);
            *reinterpret_cast<uint4*>(rowp + (((2 * c + 1) ^ (j & 7)) << 4)) = make_uint4(dk[4], dk[5], dk[6], dk[7]);
          }
          if (ok) {
            fence_proxy_async_smem();
            tc_fence_before();
            mbar_arrive(&bars[kDsReady]);
          }
        }
      }
      q0_prev = q0;
    }
    if (WANT_DBIAS && n > 0)  // the last query tile's dBias
      store_dbias(q0_prev, 0, std::integral_constant<int, 32>{});
    if (ok && n > 0) ok = mbar_wait(&bars[kFinal], 0, p.err, kDevErrTimeout, abort_flag);
    // zero-fill the dBias tiles of this key column that were skipped (TMA stores of a zero tile)
    if (WANT_DBIAS) {
      // every product has finished with the dS^T tile (kFinal): it becomes the zero tile
      reinterpret_cast<uint4*>(sDS)[ctid * 8 + 0] = make_uint4(0, 0, 0, 0);
#pragma unroll
      for (int u = 1; u < 8; ++u) reinterpret_cast<uint4*>(sDS)[ctid * 8 + u] = make_uint4(0, 0, 0, 0);
      fence_proxy_async_smem();
      named_bar_sync(1, 256);
      if (ctid == 0 && ok) {
        const uint64_t zpol = l2_evict_first();
        for (int qt = 0; qt < p.nTq; ++qt) {
          if (it.cls(qt) != kSkip) continue;
          tma_store_4d_hint(&tmDB, sDS, k0, qt * kTile, g, b, zpol);
          tma_store_4d_hint(&tmDB, sDS + 16384, k0 + 64, qt * kTile, g, b, zpol);
        }
        bulk_commit_group();
        bulk_wait_all();
      }
      named_bar_sync(1, 256);
    }
    // dK (warpgroup 0) and dV (warpgroup 1); both accumulators already carry their scale
    if (ok) {
      tc_fence_after();
      const int64_t off = ((static_cast<int64_t>(b) * p.Nk + kidx) * p.Hkv + g) * p.d;
      uint16_t* dst = (wg == 0 ? p.dk : p.dv) + off;
      const uint32_t col0 = wg == 0 ? 384u : 256u;
#pragma unroll
      for (int c = 0; c < D / 32; ++c) {
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
        if (kin) {  // columns past the head dim are padding
          uint4* d4 = reinterpret_cast<uint4*>(dst + c * 32);
#pragma unroll
          for (int v = 0; v < 4; ++v)
            if (c * 32 + v * 8 < p.d) d4[v] = make_uint4(pk[4 * v], pk[4 * v + 1], pk[4 * v + 2], pk[4 * v + 3]);
        }
      }
    }
   }
  } else {
   regs_increase<kRegsDrain>();
   if (any_active) {
    // ------------------------------------------------------------ dQ drain
    // Warp (12 + quad) reads TMEM lanes quad*32..+31 of the dQ product of every step (d = 128:
    // lane = head-dim index, columns = the 128 queries; d = 64: lane = query, columns = head
    // dim), releases the columns for the next dP^T and adds the values to the fp32 accumulator.
    const int quad = warp & 3;
    const int row = quad * 32 + lane;
    const uint32_t tl = tbase + (static_cast<uint32_t>(quad * 32) << 16);
    int n = 0;
    bool ok = true;
    for (int qt = first_qt; ok && it.valid(qt); qt = it.next(qt)) {
      const int q0 = qt * kTile;
      for (int hh = 0; hh < p.G; ++hh, ++n) {
        const int h = g * p.G + hh;
        if (!(ok = mbar_wait(&bars[kDqFull], n & 1, p.err, kDevErrTimeout, abort_flag))) break;
        tc_fence_after();
        if (DQ_T) {
          uint32_t r0[32], r1[32], r2[32], r3[32];
          tmem_ld32(tl + 128, r0);
          tmem_ld32(tl + 160, r1);
          tmem_ld32(tl + 192, r2);
          tmem_ld32(tl + 224, r3);
          tmem_ld_wait(r0);
          tmem_ld_tie(r1);
          tmem_ld_tie(r2);
          tmem_ld_tie(r3);
          tc_fence_before();
          mbar_arrive(&bars[kDqFree]);
          // The accumulator is interleaved by four queries (dq_acc_index), so each thread adds
          // four queries with one 16-byte reduction and a warp instruction covers 512
          // contiguous bytes.  The reductions are paced (kDrainPaceNs after each) so that they
          // leave the SM about as fast as the memory system accepts them: a backlog of
          // reductions stalls the other warps' shared-memory and TMEM accesses and the tensor
          // core's operand reads.
          // Head-dim rows past d are padding: a warp whose 32 rows all lie past d skips, the
          // others add all their rows (those past d hold zeros, as K's padded columns are
          // zero-filled; they land in the accumulator's padding).  A warp with only some lanes
          // active made the whole backward about 25 % slower at d = 80 or 112.
          if (quad * 32 < p.d) {
            float* dst = p.dq_acc + dq_acc_index(b, h, q0, row, p.Hq, p.nqpad, 128);
#pragma unroll
            for (int u = 0; u < 8; ++u)
              red_add_v4(dst + u * 512, __uint_as_float(r0[4 * u]), __uint_as_float(r0[4 * u + 1]),
                         __uint_as_float(r0[4 * u + 2]), __uint_as_float(r0[4 * u + 3])), __nanosleep(kDrainPaceNs);
#pragma unroll
            for (int u = 0; u < 8; ++u)
              red_add_v4(dst + (8 + u) * 512, __uint_as_float(r1[4 * u]), __uint_as_float(r1[4 * u + 1]),
                         __uint_as_float(r1[4 * u + 2]), __uint_as_float(r1[4 * u + 3])), __nanosleep(kDrainPaceNs);
#pragma unroll
            for (int u = 0; u < 8; ++u)
              red_add_v4(dst + (16 + u) * 512, __uint_as_float(r2[4 * u]), __uint_as_float(r2[4 * u + 1]),
                         __uint_as_float(r2[4 * u + 2]), __uint_as_float(r2[4 * u + 3])), __nanosleep(kDrainPaceNs);
#pragma unroll
            for (int u = 0; u < 8; ++u)
              red_add_v4(dst + (24 + u) * 512, __uint_as_float(r3[4 * u]), __uint_as_float(r3[4 * u + 1]),
                         __uint_as_float(r3[4 * u + 2]), __uint_as_float(r3[4 * u + 3])), __nanosleep(kDrainPaceNs);
          }
        } else {
          uint32_t r0[32], r1[32];
          tmem_ld32(tl + 128, r0);
          tmem_ld32(tl + 160, r1);
          tmem_ld_wait(r0);
          tmem_ld_tie(r1);
          tc_fence_before();
          mbar_arrive(&bars[kDqFree]);
          // lane = query: with the accumulator grouped by four head-dim columns, a warp's
          // reductions of one group cover 512 contiguous bytes
          float* dqrow = p.dq_acc + dq_acc_index(b, h, q0 + row, 0, p.Hq, p.nqpad, D);
          const int64_t gstep = static_cast<int64_t>(p.nqpad) * 4;  // next group of four columns
#pragma unroll
          for (int v = 0; v < 8; ++v)
            if (4 * v < p.d)
              red_add_v4(dqrow + v * gstep, __uint_as_float(r0[4 * v]), __uint_as_float(r0[4 * v + 1]),
                         __uint_as_float(r0[4 * v + 2]), __uint_as_float(r0[4 * v + 3]));
#pragma unroll
          for (int v = 0; v < 8; ++v)
            if (32 + 4 * v < p.d)
              red_add_v4(dqrow + (8 + v) * gstep, __uint_as_float(r1[4 * v]), __uint_as_float(r1[4 * v + 1]),
                         __uint_as_float(r1[4 * v + 2]), __uint_as_float(r1[4 * v + 3]));
        }
      }
    }
   }
  }
  if (WANT_DBIAS && threadIdx.x == 128) bulk_wait_all();  // compute thread 0 issued the dBias stores
  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    __syncwarp();
    tc_fence_after();
    tmem_dealloc(tbase, 512);
  }
}

template <int D, bool HB, bool WD>
cudaError_t launch_bwd_t(const CUtensorMap& tq, const CUtensorMap& tk, const CUtensorMap& tv, const CUtensorMap& tdo,
                         const CUtensorMap& tb, const CUtensorMap& tdb, const BwdParams& p, cudaStream_t stream) {
  using L = BwdSmem<D, HB>;
  auto kern = bwd_kernel<D, HB, WD>;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, L::kTotal);
  if (e != cudaSuccess) return e;
  cudaFuncAttributes fa;
  e = cudaFuncGetAttributes(&fa, kern);
  if (e != cudaSuccess) return e;
  // setmaxnreg re-balancing needs the launch allocation to cover low + 2 x high per SMSP slot
  if (fa.numRegs < kBwdMinLaunchRegs) return cudaErrorInvalidConfiguration;
  const unsigned grid = static_cast<unsigned>(p.nTk) * p.B * p.Hkv;
  kern<<<grid, kBwdThreads, L::kTotal, stream>>>(tq, tk, tv, tdo, tb, tdb, p);
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_bwd_pre(const BwdPreParams& p, cudaStream_t stream) {
  const int64_t tasks = static_cast<int64_t>(p.B) * p.Hq * ((p.nqpad + kPreRowsPerWarp - 1) / kPreRowsPerWarp);
  bwd_pre_kernel<<<static_cast<unsigned>((tasks + 7) / 8), 256, 0, stream>>>(p);
  return cudaGetLastError();
}

cudaError_t launch_dq_convert(const DqConvertParams& p, cudaStream_t stream) {
  if (p.dpad == 128) {
    const int64_t blocks = static_cast<int64_t>(p.B) * p.Hq * (p.nqpad / 4) / kCvtGroups;  // nqpad % 128 == 0
    if (blocks == 0) return cudaSuccess;
    dq_convert4_kernel<<<static_cast<unsigned>(blocks), 256, 0, stream>>>(p);
    return cudaGetLastError();
  }
  const int64_t threads = static_cast<int64_t>(p.B) * p.Hq * (p.dpad >> 3) * p.nqpad;
  if (threads == 0) return cudaSuccess;
  dq_convert_grouped_kernel<<<static_cast<unsigned>((threads + 255) / 256), 256, 0, stream>>>(p);
  return cudaGetLastError();
}

cudaError_t launch_bwd(int d, bool has_bias, bool want_dbias, const CUtensorMap& tq, const CUtensorMap& tk,
                       const CUtensorMap& tv, const CUtensorMap& tdo, const CUtensorMap& tb, const CUtensorMap& tdb,
                       const BwdParams& p, cudaStream_t stream) {
  if (d == 128) {
    if (want_dbias) return launch_bwd_t<128, true, true>(tq, tk, tv, tdo, tb, tdb, p, stream);
    return has_bias ? launch_bwd_t<128, true, false>(tq, tk, tv, tdo, tb, tdb, p, stream)
                    : launch_bwd_t<128, false, false>(tq, tk, tv, tdo, tb, tdb, p, stream);
  }
  if (d == 64) {
    if (want_dbias) return launch_bwd_t<64, true, true>(tq, tk, tv, tdo, tb, tdb, p, stream);
    return has_bias ? launch_bwd_t<64, true, false>(tq, tk, tv, tdo, tb, tdb, p, stream)
                    : launch_bwd_t<64, false, false>(tq, tk, tv, tdo, tb, tdb, p, stream);
  }
  return cudaErrorInvalidValue;
}

}  // namespace fdma
