// Parameter blocks and launcher declarations shared by the host layer
// (fdma_api.cu) and the kernel translation units.
#pragma once

#include <cstddef>
#include <cstdint>
#include <cuda.h>
#include <cuda_runtime.h>

#include "../../include/fdma.h"

namespace fdma {

constexpr int kTile = 128;           // query rows and key columns per tile
constexpr int kMaxKTiles = 1024;     // Nk <= 131072
constexpr int kTopkMaxKeys = 65536;  // one row's keys held in shared memory

// Head dims 64 and 72..128 (multiples of 8).  A head dim between 64 and 128 runs on the
// kernels for 128: the TMA load of its upper 64-column box zero-fills the columns past d,
// which then add nothing to any product, and nothing is stored past column d.  (Head dims
// below 64 would need 64-byte-swizzled tiles: the 64-column box cannot be wider than the
// tensor.)
inline int padded_head_dim(int d) { return d <= 64 ? 64 : 128; }
// Head dims: multiples of 8 from 8 to 128.  The kernels are built for 64 and 128; a smaller
// head dim runs on the next one up, the missing columns of Q, K, V and dO read as zeros by TMA
// (out-of-range fill) and the padding columns of the results never stored.
inline bool head_dim_ok(int d) { return d >= 8 && d <= 128 && d % 8 == 0; }
// Head dim of v, out and dout: fdma_args.dv, 0 meaning the q/k head dim d.
inline int head_dim_v(const fdma_args& a) { return a.dv > 0 ? a.dv : a.d; }
// d = dv from 8 to 128 (the 64- / 128-wide kernels), or (d, dv) = (192, 128) or (256, 256)
// (the wide one-head forward and the output-split backward).
inline bool head_dims_ok(int d, int dv) {
  return (head_dim_ok(d) && dv == d) || (d == 192 && dv == 128) || (d == 256 && dv == 256);
}
// Row width of the fp32 dQ accumulator: the padded width up to 128, else d itself.
inline int dq_acc_width(int d) { return d <= 128 ? padded_head_dim(d) : d; }
constexpr int kSkip = 0, kPartial = 1, kFull = 2;

// Device error word values (first writer wins).
constexpr int kDevErrTimeout = FDMA_ERR_TIMEOUT;
constexpr int kDevErrAlign = FDMA_ERR_CUDA;

// One 128x128 tile's keep-bits: 128 x 16 bytes.  bits_row[t*128 + r] holds
// row r (bit c%32 of word c/32 = column c); bits_col[t*128 + c] holds column c
// (bit r%32 of word r/32 = row r).
struct ClassifyParams {
  int B, Nq, Nk, Hkv, nTq, nTk;
  int mask_kind, causal, no_skip;
  int causal_off;  // key j is visible from query i when j <= i + causal_off (Nk - Nq, or q_offset)
  int mask_bsel, mask_hsel;  // bf16 masks by TMA: 0 where the mask is broadcast (coordinate 0)
  int* err;                  // device error word (the TMA classifier's bounded wait)
  const uint16_t* mask;
  const uint8_t* mask_u8;  // same buffer, FDMA_MASK_DENSE_U8 / FDMA_MASK_BITS
  int64_t ms_b, ms_h, ms_r;
  const int32_t* cr;
  int64_t cr_b, cr_h;
  int8_t* kmap;      // kernel tile classes (workspace)
  int8_t* user_map;  // optional caller copy of the true classes
  uint4* bits_row;
  uint4* bits_col;
};

struct FwdParams {
  int B, Nq, Nk, Hq, Hkv, G, nTq, nTk;
  int d;   // head dim of q, k (up to 128 the kernel runs on its padded width, 64 or 128)
  int dv;  // head dim of v, out (= d up to 128)
  int bias_bsel, bias_hsel;  // 0 where the bias is broadcast over batch / kv head (TMA coordinate 0)
  float scale, scale_log2;  // softmax scale and scale * log2(e)
  int test_short_wait;      // FDMA_FLAG_TEST_SHORT_WAIT: the softmax warps time out on purpose
  const int8_t* kmap;
  const uint4* bits_row;
  uint16_t* out;  // (B,Nq,Hq,d)
  float* lse;     // (B,Hq,Nq)
  int* err;
};

struct BwdPreParams {
  int B, Nq, Hq, d, nqpad;
  int dpad;     // row width of the dQ accumulator (64 or 128)
  float scale;  // softmax scale
  const uint16_t* out;
  const uint16_t* dout;
  const float* lse;
  float* lse2;   // (B,Hq,nqpad): -lse*log2(e), -inf for empty / padded rows
  float* delta;  // (B,Hq,nqpad): -scale * <dO_i, O_i>
  float* dq_acc; // dQ accumulator (layout: dq_acc_index), zeroed
};

// fp32 dQ accumulator of the backward.  For the 128-wide kernels it is interleaved by
// groups of four query rows, (B, Hq, nqpad/4, 128, 4): element (query i, head-dim c) of a
// head sits at ((i/4)*128 + c)*4 + i%4, so the four queries of one head-dim index are one
// 16-byte vector and 32 consecutive head-dim indices are 512 contiguous bytes.  For the
// 64-wide kernels and the wide head dims (a TMEM lane holds a query there) it is grouped by
// four head-dim columns, (B, Hq, dpad/4, nqpad, 4): the four columns of one query are one
// 16-byte vector and 32 consecutive queries are 512 contiguous bytes.
__host__ __device__ inline int64_t dq_acc_index(int b, int h, int i, int c, int Hq, int nqpad, int dpad) {
  if (dpad == 128)
    return (((static_cast<int64_t>(b) * Hq + h) * (nqpad >> 2) + (i >> 2)) * 128 + c) * 4 + (i & 3);
  return (((static_cast<int64_t>(b) * Hq + h) * (dpad >> 2) + (c >> 2)) * nqpad + i) * 4 + (c & 3);
}

struct BwdParams {
  int B, Nq, Nk, Hq, Hkv, G, nTq, nTk, nqpad;
  int d;  // head dim of q, k, v, dout, dk, dv (the kernel runs on its padded width)
  int bias_bsel, bias_hsel;  // 0 where the bias is broadcast over batch / kv head (TMA coordinate 0)
  float scale, scale_log2;
  int test_short_wait;  // FDMA_FLAG_TEST_SHORT_WAIT: the compute warps time out on purpose
  const int8_t* kmap;
  const uint4* bits_col;
  const uint16_t* bias;  // may be null
  int64_t bs_b, bs_h, bs_r;
  const float* lse2;
  const float* delta;
  float* dq_acc;
  uint16_t* dk;     // (B,Nk,Hkv,d)
  uint16_t* dv;     // (B,Nk,Hkv,d)
  uint16_t* dbias;  // (B,Hkv,Nq,Nk) or null
  int* err;
};

struct DqConvertParams {
  int B, Nq, Hq, d, nqpad;
  int dpad;  // row width of the dQ accumulator
  const float* dq_acc;
  uint16_t* dq;
};

// Workspace layout (byte offsets, each 256-aligned).
struct WorkspaceLayout {
  size_t kmap, bits_row, bits_col, lse2, delta, dq_acc, total_fwd, total_bwd;
};

WorkspaceLayout workspace_layout(int B, int Nq, int Nk, int Hq, int Hkv, int d);

struct TopkParams {
  int B, Hkv, Nq, Nk, keep;
  int64_t bias_stride[3];  // elements: batch, kv head, row (the key dimension is contiguous)
  const uint16_t* bias;    // bf16
  uint16_t* bias_out;      // bf16 with bias_stride, or nullptr; may equal bias
  uint16_t* mask_bf16;     // (B,Hkv,Nq,Nk) contiguous, or nullptr
  uint8_t* mask_u8;        // (B,Hkv,Nq,Nk) contiguous, or nullptr
};

cudaError_t launch_classify(const ClassifyParams& p, cudaStream_t stream);
// bf16 masks through a tensor map of the mask (4D, 64 x 128 box, 128-byte swizzle).
cudaError_t launch_classify_tma1(const CUtensorMap& tm, const ClassifyParams& p, cudaStream_t stream);
cudaError_t launch_topk(const TopkParams& p, cudaStream_t stream);
size_t topk_smem_bytes(int Nk);
cudaError_t launch_fwd(int d, int dv, bool has_bias, const CUtensorMap& tq, const CUtensorMap& tk, const CUtensorMap& tv,
                       const CUtensorMap& tb, const FwdParams& p, cudaStream_t stream);
cudaError_t launch_bwd_pre(const BwdPreParams& p, cudaStream_t stream);
// (d, dv) = (192, 128) or (256, 256): both output parts, dBias from the first.
cudaError_t launch_bwd_wide(int d, int dv, bool has_bias, bool want_dbias, const CUtensorMap& tq,
                            const CUtensorMap& tk, const CUtensorMap& tv, const CUtensorMap& tdo,
                            const CUtensorMap& tb, const BwdParams& p, cudaStream_t stream);
cudaError_t launch_bwd(int d, bool has_bias, bool want_dbias, const CUtensorMap& tq, const CUtensorMap& tk,
                       const CUtensorMap& tv, const CUtensorMap& tdo, const CUtensorMap& tb, const CUtensorMap& tdb,
                       const BwdParams& p, cudaStream_t stream);
cudaError_t launch_dq_convert(const DqConvertParams& p, cudaStream_t stream);

}  // namespace fdma
